"""Layer streaming through afx_stream_run: compressed layers copied from pinned
host memory while earlier layers decode; every output checked against the
oracle."""
import numpy as np
import pytest

import oracle
from afx_testutil import within_gemv_tolerance
from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu


def _layer(afx, seed, shapes):
    """Containers of one small layer packed into one blob, with their ops."""
    import torch
    parts, metas, off = [], [], 0
    for i, (kind, shape) in enumerate(shapes):
        n = int(np.prod(shape))
        w = synth.normal(n, 1.0 if kind == "norm" else 0.0, 0.05 if kind == "norm" else 0.02, seed=seed, stream=i)
        c, d = afx.encode(w)
        parts.append(c)
        metas.append((kind, shape, w, c, d, off))
        off += c.size
    blob = torch.empty(off, dtype=torch.uint8).pin_memory()
    blob.numpy()[:] = np.concatenate(parts)
    return blob, metas


def _ops(afx, metas, B, keep):
    import torch
    ops = []
    for kind, shape, w, c, d, off in metas:
        op = afx.afx_op()
        op.desc = d
        op.offset = off
        if kind == "norm" or kind == "decode":
            out = torch.empty(d.n, dtype=torch.int16, device="cuda")
            op.kind = afx.AFX_OP_DECODE
            op.out_dev = out.data_ptr()
            keep.append(("decode", out, w, None))
        else:
            rows, cols = shape
            x = synth.activations(B, cols, seed=rows)
            xd = torch.from_numpy(x.view(np.int16)).cuda()
            y = torch.full((B, rows), float("nan"), dtype=torch.float32, device="cuda")
            ws = torch.empty(afx.afx_decode_gemv_workspace(d, B) // 4 + 4, dtype=torch.float32, device="cuda")
            op.kind = afx.AFX_OP_GEMV
            op.rows, op.cols, op.batch = rows, cols, B
            op.x_dev, op.out_dev, op.workspace_dev = xd.data_ptr(), y.data_ptr(), ws.data_ptr()
            op.workspace_bytes = ws.numel() * 4
            keep.append(("gemv", y, (w, c, x, rows, cols), (xd, ws)))
        ops.append(op)
    return ops


@pytest.mark.parametrize("n_bufs", [2, 3])
def test_streamed_layers_match_the_oracle(afx, n_bufs):
    import torch
    shapes = [("norm", (640,)), ("gemv", (96, 640)), ("gemv", (640, 1024)), ("decode", (256, 640)),
              ("norm", (640,)), ("gemv", (1024, 640))]
    keep, layers = [], []
    for l in range(5):
        blob, metas = _layer(afx, 100 + l, shapes)
        layers.append((blob, _ops(afx, metas, 1 + l % 4, keep)))
    buf_bytes = max(b.numel() for b, _ in layers)
    bufs = [torch.empty(buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(n_bufs)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy = torch.cuda.Stream()
    afx.afx_stream_run(layers, bufs, buf_bytes, torch.cuda.current_stream(), copy, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for kind, out, ref, _ in keep:
        if kind == "decode":
            assert np.array_equal(out.cpu().numpy().view(np.uint16), ref)
        else:
            w, c, x, rows, cols = ref
            y_ref, A = oracle.gemv(w.reshape(rows, cols), x)
            assert within_gemv_tolerance(out.cpu().numpy(), y_ref, A)


def test_one_device_output_shared_by_every_layer_copied_back(afx):
    # every layer restores into the same device buffer and copies it back to
    # its own host buffer: each layer's op must wait until the previous
    # layer's copy back has read the buffer, and two calls in a row reuse it
    import torch
    layers, refs, hosts = [], [], []
    n_max = 400_000
    shared = torch.empty(n_max, dtype=torch.int16, device="cuda")
    for l in range(6):
        w = synth.normal(n_max - 7_919 * l, seed=70 + l)
        c, d = afx.encode(w)
        blob = torch.empty(c.size, dtype=torch.uint8).pin_memory()
        blob.numpy()[:] = c
        host = torch.full((d.n,), -1, dtype=torch.int16).pin_memory()
        op = afx.afx_op()
        op.desc, op.offset, op.kind = d, 0, afx.AFX_OP_DECODE
        op.out_dev, op.out_host = shared.data_ptr(), host.data_ptr()
        layers.append((blob, [op]))
        refs.append(w)
        hosts.append(host)
    buf_bytes = max(b.numel() for b, _ in layers)
    bufs = [torch.empty(buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(2):
        for h in hosts:
            h.fill_(-1)
        afx.afx_stream_run(layers, bufs, buf_bytes, torch.cuda.current_stream(), copy, status_dev=status,
                           d2h_stream=d2h)
        afx.afx_stream_run(layers[::-1], bufs, buf_bytes, torch.cuda.current_stream(), copy, status_dev=status,
                           d2h_stream=d2h)
        torch.cuda.synchronize()
        assert status.item() == 0
        for w, host in zip(refs, hosts):
            assert np.array_equal(host.numpy().view(np.uint16), w)


@pytest.mark.parametrize("own_stream", [False, True])
def test_restored_tensors_copied_back_to_host(afx, own_stream):
    # one tensor per layer, each restored on the GPU and copied back to pinned host memory
    import torch
    layers, refs, hosts = [], [], []
    for l in range(6):
        w = synth.normal(50_000 + 9_999 * l, seed=40 + l)
        c, d = afx.encode(w)
        blob = torch.empty(c.size, dtype=torch.uint8).pin_memory()
        blob.numpy()[:] = c
        out = torch.empty(d.n, dtype=torch.int16, device="cuda")
        host = torch.full((d.n,), -1, dtype=torch.int16).pin_memory()
        op = afx.afx_op()
        op.desc, op.offset, op.kind = d, 0, afx.AFX_OP_DECODE
        op.out_dev, op.out_host = out.data_ptr(), host.data_ptr()
        layers.append((blob, [op]))
        refs.append((w, out))
        hosts.append(host)
    buf_bytes = max(b.numel() for b, _ in layers)
    bufs = [torch.empty(buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy = torch.cuda.Stream()
    d2h = torch.cuda.Stream() if own_stream else None
    afx.afx_stream_run(layers, bufs, buf_bytes, torch.cuda.current_stream(), copy, status_dev=status, d2h_stream=d2h)
    torch.cuda.synchronize()
    assert status.item() == 0
    for (w, out), host in zip(refs, hosts):
        assert np.array_equal(host.numpy().view(np.uint16), w)


def test_streamed_mixed_formats_copied_back_to_host(afx):
    # layers of BF16, FP16 and E4M3 tensors (several per layer, one batch
    # launch per format), each restored and copied back to pinned host memory
    import torch
    gens = [(0, lambda n, s: synth.normal(n, seed=s)), (1, lambda n, s: synth.normal_fp16(n, seed=s)),
            (2, lambda n, s: synth.normal_e4m3(n, seed=s))]
    layers, refs = [], []
    for l in range(4):
        parts, ops, off = [], [], 0
        for k, (fmt, gen) in enumerate(gens):
            w = gen(30_001 + 7_777 * l + 1_111 * k, 60 + 3 * l + k)
            c, d = afx.encode(w, fmt=fmt)
            dt = torch.uint8 if fmt == 2 else torch.int16
            out = torch.empty(d.n, dtype=dt, device="cuda")
            host = torch.full((d.n,), 0x5A if fmt == 2 else -1, dtype=dt).pin_memory()
            op = afx.afx_op()
            op.desc, op.offset, op.kind = d, off, afx.AFX_OP_DECODE
            op.out_dev, op.out_host = out.data_ptr(), host.data_ptr()
            parts.append(c)
            ops.append(op)
            refs.append((fmt, w, out, host))
            off += c.size
        blob = torch.empty(off, dtype=torch.uint8).pin_memory()
        blob.numpy()[:] = np.concatenate(parts)
        layers.append((blob, ops))
    buf_bytes = max(b.numel() for b, _ in layers)
    bufs = [torch.empty(buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    compute = torch.cuda.current_stream()
    afx.afx_stream_run(layers, bufs, buf_bytes, compute, copy, status_dev=status, d2h_stream=d2h)
    st, word = afx.afx_sync(d2h, 30_000, status)
    torch.cuda.synchronize()
    assert (st, word) == (afx.AFX_OK, 0)
    for fmt, w, out, host in refs:
        got = host.numpy()
        assert np.array_equal(got if fmt == 2 else got.view(np.uint16), w), fmt


def test_blob_larger_than_buffer_is_rejected(afx):
    import torch
    blob, metas = _layer(afx, 7, [("decode", (64, 640))])
    keep = []
    ops = _ops(afx, metas, 1, keep)
    bufs = [torch.empty(256, dtype=torch.uint8, device="cuda") for _ in range(2)]
    with pytest.raises(afx.AfxError):
        afx.afx_stream_run([(blob, ops)], bufs, 256)


@pytest.mark.slow
@pytest.mark.parametrize("B", [1, 4])
def test_forty_streamed_full_size_layers_against_the_oracle(afx, B):
    # the bench's streaming configuration: four distinct Qwen3-14B-shaped
    # layers in pinned host memory cycle over 40 streamed layers, norms
    # restored and the seven matrices through the fused GEMV.  Every layer's
    # norms are checked bit for bit; the first layer's products row by row
    # against the oracle's GEMV, and 16 sampled rows of every other product
    # against the oracle's GEMV of those rows
    import torch
    import bench
    blobs = []
    for seed in range(4):
        parts = bench.build_layer(seed, 0, "layer")
        size = sum(c.size for _, _, c, _ in parts)
        blob = torch.empty(size, dtype=torch.uint8).pin_memory()
        o = 0
        for _, _, c, _ in parts:
            blob.numpy()[o:o + c.size] = c
            o += c.size
        blobs.append((blob, parts))
    keep, layers, outs = [], [], []
    for l in range(40):
        blob, parts = blobs[l % len(blobs)]
        first = len(keep)
        ops = bench._layer_ops(afx, parts, B, torch.device("cuda"), keep)
        layers.append((blob, ops))
        outs.append(keep[first:])
    buf_bytes = max(b.numel() for b, _ in blobs)
    bufs = [torch.empty(buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_stream_run(layers, bufs, buf_bytes, torch.cuda.current_stream(), torch.cuda.Stream(), status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    shapes = {name: shape for name, shape, _ in synth.LAYER_TENSORS}
    rng = np.random.default_rng(B)
    for l in range(40):
        _, parts = blobs[l % len(blobs)]
        it = iter(outs[l])
        for name, w, _, _ in parts:
            if len(shapes[name]) == 1:  # a norm vector, restored
                assert np.array_equal(next(it).cpu().numpy().view(np.uint16), w.reshape(-1))
                continue
            x_t, y_t, _ = next(it), next(it), next(it)
            rows, cols = shapes[name]
            x = x_t.cpu().numpy().view(np.uint16).reshape(B, cols)
            y = y_t.cpu().numpy()
            W = w.reshape(rows, cols)
            pick = np.arange(rows) if l == 0 else np.sort(rng.choice(rows, size=16, replace=False))
            y_ref, A = oracle.gemv(np.ascontiguousarray(W[pick]), x)
            assert within_gemv_tolerance(y[:, pick], y_ref, A), (l, name)
