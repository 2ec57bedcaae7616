"""GPU restore of the other element formats (FP16, E4M3) through the C ABI,
bit for bit against the CPU oracle: ragged sizes, every bit pattern, the
single-symbol fill, both decode paths (byte-step table and 12-bit table),
host-resident containers, mixed-format batches, corrupt streams, and the
calls that take BF16 only."""
import numpy as np
import pytest

import oracle
from afx_testutil import gpu_decode_any
from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu

FP16, E4M3 = 1, 2


def _check(afx, w, fmt, chunk_bytes=0, **kw):
    w = np.ascontiguousarray(w).reshape(-1)
    c, d = afx.encode(w, chunk_bytes=chunk_bytes, fmt=fmt)
    ref, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(ref, w)
    out, status, intact = gpu_decode_any(afx, c, d, **kw)
    assert status == 0
    assert intact, "wrote outside the output range"
    mism = np.flatnonzero(out != ref)
    assert mism.size == 0, f"{mism.size} mismatches, first at {mism[:5]}"
    return c, d


@pytest.mark.parametrize("n", [1, 2, 3, 15, 16, 17, 31, 33, 255, 257, 1000, 4097, 65_537, 300_007, 1_000_003])
def test_e4m3_ragged_sizes(afx, n):
    c, d = _check(afx, synth.normal_e4m3(n, seed=n), E4M3, out_pad=40, out_offset=16)
    assert d.format == E4M3


@pytest.mark.parametrize("n", [1, 7, 9, 1000, 65_537, 1_000_003])
def test_fp16_ragged_sizes(afx, n):
    _check(afx, synth.normal_fp16(n, seed=n), FP16, out_pad=24)


@pytest.mark.parametrize("T", [4, 8, 16])
def test_e4m3_every_pattern_every_chunk_size(afx, T):
    rng = np.random.default_rng(T)
    w = np.concatenate([rng.permutation(synth.all_e4m3_patterns()) for _ in range(300)])
    _check(afx, w, E4M3, chunk_bytes=T, out_pad=16)


@pytest.mark.parametrize("T", [4, 16])
def test_fp16_every_pattern(afx, T):
    w = synth.all_bf16_patterns()
    rng = np.random.default_rng(T)
    _check(afx, np.concatenate([w, rng.permutation(w)]), FP16, chunk_bytes=T)


def test_e4m3_byte_step_path_and_12_bit_path(afx):
    # an even spread of exponents: shortest code >= 2 bits (byte-step table);
    # one dominant exponent: a 1-bit code (12-bit table)
    even = synth.normal_e4m3(500_003, seed=21)
    c, d = _check(afx, even, E4M3, out_pad=16)
    assert min(l for l in d.len if l) >= 2
    rng = np.random.default_rng(22)
    dom = np.where(rng.random(400_001) < 0.7, np.uint8(0x38), even[:400_001])
    c, d = _check(afx, dom, E4M3, out_pad=16)
    assert min(l for l in d.len if l) == 1


@pytest.mark.parametrize("n", [1, 15, 16, 17, 100_001])
def test_e4m3_single_exponent_fill(afx, n):
    w = np.resize(synth.e4m3_round(np.array([1.0, -1.125, 1.5, -1.875, 1.25], np.float32)), n)
    c, d = _check(afx, w, E4M3, out_pad=16, out_offset=16)
    assert d.nsym == 1 and d.fill == 7


def test_fp16_norm_vector_and_single(afx):
    _check(afx, synth.normal_fp16(5120, 1.0, 0.05, seed=3), FP16)
    _check(afx, np.full(1001, 0x3C00, np.uint16), FP16)


def test_e4m3_host_resident_container(afx):
    w = synth.normal_e4m3(700_001, seed=23)
    c, d = afx.encode(w, fmt=E4M3)
    out, status, intact = gpu_decode_any(afx, c, d, out_pad=16, host=True)
    assert status == 0 and intact and np.array_equal(out, w)


def test_mixed_format_batch(afx):
    import torch
    tensors = [(synth.normal(300_001, seed=31), 0), (synth.normal_fp16(200_003, seed=32), FP16),
               (synth.normal_e4m3(500_001, seed=33), E4M3), (np.full(77, 0x38, np.uint8), E4M3),
               (synth.normal_e4m3(17, seed=34), E4M3), (synth.normal(5120, 1.0, 0.05, seed=35), 0)]
    descs, conts, outs = [], [], []
    for w, fmt in tensors:
        c, d = afx.encode(w, fmt=fmt)
        descs.append(d)
        conts.append(torch.from_numpy(c).cuda())
        outs.append(torch.zeros(w.size, dtype=torch.uint8 if fmt == E4M3 else torch.int16, device="cuda"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_batch(descs, conts, outs, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for (w, fmt), o in zip(tensors, outs):
        got = o.cpu().numpy()
        assert np.array_equal(got if fmt == E4M3 else got.view(np.uint16), w)


def test_e4m3_corrupt_stream_is_flagged(afx):
    import torch
    w = synth.normal_e4m3(400_000, seed=36)
    c, d = afx.encode(w, fmt=E4M3)
    rng = np.random.default_rng(9)
    bad = c.copy()
    bad[d.off_exp: d.off_exp + d.n_chunks * d.chunk_bytes] = rng.integers(0, 256, d.n_chunks * d.chunk_bytes,
                                                                          dtype=np.uint8)
    out = torch.zeros(w.size + 64, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode(d, torch.from_numpy(bad).cuda(), out[:w.size], status_dev=status)
    torch.cuda.synchronize()
    assert status.item() != 0
    assert not out[w.size:].cpu().numpy().any()  # nothing written past the output


def test_output_element_size_must_match_the_format(afx):
    import torch
    w = synth.normal_e4m3(1000, seed=37)
    c, d = afx.encode(w, fmt=E4M3)
    with pytest.raises(ValueError):
        afx.afx_decode(d, torch.from_numpy(c).cuda(), torch.zeros(1000, dtype=torch.int16, device="cuda"))


def test_gemv_and_prefill_refuse_other_formats(afx):
    import torch
    rows, cols = 64, 2048
    x = torch.zeros((1, cols), dtype=torch.int16, device="cuda")
    y = torch.zeros((1, rows), dtype=torch.float32, device="cuda")
    for w, fmt in ((synth.normal_fp16(rows * cols, seed=1), FP16), (synth.normal_e4m3(rows * cols, seed=1), E4M3)):
        c, d = afx.encode(w, fmt=fmt)
        dev = torch.from_numpy(c).cuda()
        ws = torch.empty(afx.afx_decode_gemv_workspace(d, 1) // 4 + 4, dtype=torch.float32, device="cuda")
        with pytest.raises(afx.AfxError):
            afx.afx_decode_gemv(d, dev, rows, cols, x, y, ws)
    c, d = afx.encode(synth.normal_e4m3(rows * cols, seed=2), fmt=E4M3)
    gws = torch.empty(afx.AFX_PREFILL_GEMM_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    with pytest.raises(afx.AfxError):
        afx.afx_prefill(d, torch.from_numpy(c).cuda(), rows, cols, torch.zeros((4, cols), dtype=torch.int16,
                        device="cuda"), torch.zeros((4, rows), dtype=torch.float32, device="cuda"),
                        torch.empty(rows * cols, dtype=torch.int16, device="cuda"), gws)


@pytest.mark.parametrize("n_tokens", [1, 33, 128])
def test_fp16_prefill_matches_float64(afx, n_tokens):
    import torch
    rows, cols = 320, 2560
    W = synth.normal_fp16(rows * cols, seed=41).reshape(rows, cols)
    X = synth.fp16_round(np.random.default_rng(42).standard_normal((n_tokens, cols)).astype(np.float32))
    c, d = afx.encode(W.reshape(-1), fmt=FP16)
    y = torch.full((n_tokens, rows), float("nan"), dtype=torch.float32, device="cuda")
    scratch = torch.empty(rows * cols, dtype=torch.int16, device="cuda")
    ws = torch.empty(afx.AFX_PREFILL_GEMM_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_prefill(d, torch.from_numpy(c).cuda(), rows, cols, torch.from_numpy(X.view(np.int16)).cuda(), y, scratch,
                    ws, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(scratch.cpu().numpy().view(np.uint16), W.reshape(-1))
    Wf = W.view(np.float16).astype(np.float64)
    Xf = X.view(np.float16).astype(np.float64)
    ref, A = Xf @ Wf.T, np.abs(Xf) @ np.abs(Wf).T
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= 2e-3 * A + np.abs(ref) * 2.0 ** -23)


@pytest.mark.slow
def test_e4m3_and_fp16_layer_matrices_full_size(afx):
    # the Qwen3-14B-shaped layer's seven matrices in each format, one batch launch, bit-exact
    import torch
    for fmt in (E4M3, FP16):
        ws, descs, conts, outs = [], [], [], []
        for name, shape, kind in synth.LAYER_TENSORS:
            if kind != "matrix":
                continue
            w = (synth.layer_matrix_e4m3(name) if fmt == E4M3 else synth.layer_tensor_fp16(name)).reshape(-1)
            c, d = afx.encode(w, fmt=fmt)
            ws.append(w)
            descs.append(d)
            conts.append(torch.from_numpy(c).cuda())
            outs.append(torch.empty(w.size, dtype=torch.uint8 if fmt == E4M3 else torch.int16, device="cuda"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        afx.afx_decode_batch(descs, conts, outs, status_dev=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        for w, o in zip(ws, outs):
            got = o.cpu().numpy()
            assert np.array_equal(got if fmt == E4M3 else got.view(np.uint16), w)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 15, 16, 17, 1001])
def test_fp16_single_exponent_fill_with_hi_bits(afx, n):
    # every element in [1, 2): one exponent (15), all fraction bits in use
    rng = np.random.default_rng(n)
    w = (np.uint16(0x3C00) | rng.integers(0, 1024, size=n).astype(np.uint16)) ^ (
        rng.integers(0, 2, size=n).astype(np.uint16) << np.uint16(15))
    c, d = _check(afx, w, FP16, out_pad=16, out_offset=8)
    assert d.nsym == 1 and d.fill == 15


@pytest.mark.parametrize("T", [4, 8])
def test_fp16_small_chunks_ragged(afx, T):
    _check(afx, synth.normal_fp16(300_007, seed=T), FP16, chunk_bytes=T, out_pad=24)


def test_fp16_host_resident_container(afx):
    w = synth.normal_fp16(500_003, seed=29)
    c, d = afx.encode(w, fmt=FP16)
    out, status, intact = gpu_decode_any(afx, c, d, out_pad=16, host=True)
    assert status == 0 and intact and np.array_equal(out, w)


def test_fp16_every_hi_pattern_at_every_position(afx):
    # every hi value in both nibbles of a byte and at every element of a
    # group of 8 (the merge's word), with groups split at both range ends
    vals = np.array([(e << 10) | (h << 7) | m for e in (13, 14, 15, 16) for h in range(8) for m in (0, 5, 127)],
                    np.uint16)
    w = np.resize(np.random.default_rng(3).permutation(vals), 8 * 97 + 5)
    _check(afx, w, FP16, out_pad=16)
