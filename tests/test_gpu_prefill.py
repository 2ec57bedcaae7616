"""Prefill products (afx_prefill, afx_prefill_batch): the container restored
into scratch memory and multiplied by the tensor cores, checked against the
oracle's GEMV (float64 products and sums of the original BF16 weights, one
token vector per batch row), |err| <= 2e-3 * sum|w x| per output (float32
accumulation over up to 17,408 terms)."""
import numpy as np
import pytest

import oracle
from afx_testutil import within_gemv_tolerance
from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu


def _within(y, W, X):
    """y [tokens][rows] against oracle.gemv(W, X): (within tolerance, worst error / sum|w x|)."""
    y_ref, A = oracle.gemv(np.ascontiguousarray(W), np.ascontiguousarray(X))
    err = np.abs(y.astype(np.float64) - y_ref.astype(np.float64))
    return within_gemv_tolerance(y, y_ref, A), float(np.max(err / np.maximum(A, 1e-30)))


def _bufs(afx, rows, cols, n_tokens):
    import torch
    y = torch.full((n_tokens, rows), float("nan"), dtype=torch.float32, device="cuda")
    scratch = torch.empty(rows * cols, dtype=torch.int16, device="cuda")
    ws = torch.empty(afx.AFX_PREFILL_GEMM_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    return y, scratch, ws


@pytest.mark.parametrize("shape", [(256, 5120), (1024, 640), (100, 4096), (33, 17408)])
@pytest.mark.parametrize("n_tokens", [1, 17, 128])
def test_prefill_matches_float64(afx, shape, n_tokens):
    import torch
    rows, cols = shape
    W = synth.normal(rows * cols, seed=rows + n_tokens).reshape(rows, cols)
    X = synth.activations(n_tokens, cols, seed=cols)
    c, d = afx.encode(W.reshape(-1))
    y, scratch, ws = _bufs(afx, rows, cols, n_tokens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_prefill(d, torch.from_numpy(c).cuda(), rows, cols, torch.from_numpy(X.view(np.int16)).cuda(), y, scratch,
                    ws, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(scratch.cpu().numpy().view(np.uint16), W.reshape(-1))  # the restored weights
    ok, worst = _within(y.cpu().numpy(), W, X)
    assert ok, worst


def test_prefill_batch_overlapped_twice(afx):
    import torch
    shapes = [(512, 1024), (128, 5120), (640, 640), (64, 4096), (256, 2048)]
    n_tokens = 64
    items = []
    for i, (r, cl) in enumerate(shapes):
        W = synth.normal(r * cl, seed=400 + i).reshape(r, cl)
        X = synth.activations(n_tokens, cl, seed=500 + i)
        c, d = afx.encode(W.reshape(-1))
        items.append((W, X, torch.from_numpy(c).cuda(), d, torch.from_numpy(X.view(np.int16)).cuda()))
    biggest = max(r * cl for r, cl in shapes)
    scratch = [torch.empty(biggest, dtype=torch.int16, device="cuda") for _ in range(2)]
    ws = torch.empty(afx.AFX_PREFILL_GEMM_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    rs, gs = torch.cuda.Stream(), torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the second call reuses the scratch buffers the first one filled
        ys = [torch.full((n_tokens, r), float("nan"), dtype=torch.float32, device="cuda") for r, _ in shapes]
        afx.afx_prefill_batch([it[3] for it in items], [it[2] for it in items], shapes, [it[4] for it in items], ys,
                              scratch, ws, restore_stream=rs, gemm_stream=gs, status_dev=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        for (W, X, *_), y in zip(items, ys):
            ok, worst = _within(y.cpu().numpy(), W, X)
            assert ok, worst


def test_prefill_batch_one_restore_launch(afx):
    import torch
    shapes = [(512, 1024), (128, 5120), (33, 640), (64, 4096), (1, 2064)]
    n_tokens = 40
    items = []
    for i, (r, cl) in enumerate(shapes):
        W = synth.normal(r * cl, seed=600 + i).reshape(r, cl)
        X = synth.activations(n_tokens, cl, seed=700 + i)
        c, d = afx.encode(W.reshape(-1))
        items.append((W, X, torch.from_numpy(c).cuda(), d, torch.from_numpy(X.view(np.int16)).cuda()))
    # each matrix starts at a 256-byte boundary of the one scratch buffer
    total = sum((2 * r * cl + 255) // 256 * 256 for r, cl in shapes) // 2
    scratch = torch.full((total,), -1, dtype=torch.int16, device="cuda")
    ws = torch.empty(afx.AFX_PREFILL_GEMM_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    gs = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = [torch.full((n_tokens, r), float("nan"), dtype=torch.float32, device="cuda") for r, _ in shapes]
    afx.afx_prefill_batch([it[3] for it in items], [it[2] for it in items], shapes, [it[4] for it in items], ys,
                          [scratch, None], ws, gemm_stream=gs, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    flat = scratch.cpu().numpy().view(np.uint16)
    off = 0
    for (W, X, *_), y, (r, cl) in zip(items, ys, shapes):
        assert np.array_equal(flat[off: off + r * cl], W.reshape(-1))
        assert np.all(flat[off + r * cl: off + (2 * r * cl + 255) // 256 * 128] == 0xFFFF)  # padding untouched
        off += (2 * r * cl + 255) // 256 * 128
        ok, worst = _within(y.cpu().numpy(), W, X)
        assert ok, worst


def test_prefill_bad_arguments(afx):
    import torch
    rows, cols = 64, 256
    c, d = afx.encode(synth.normal(rows * cols, seed=1))
    y, scratch, ws = _bufs(afx, rows, cols, 4)
    x = torch.zeros((4, cols), dtype=torch.int16, device="cuda")
    dev = torch.from_numpy(c).cuda()
    with pytest.raises(afx.AfxError):
        afx.afx_prefill(d, dev, rows + 1, cols, torch.zeros((4, cols), dtype=torch.int16, device="cuda"),
                        torch.zeros((4, rows + 1), dtype=torch.float32, device="cuda"),
                        torch.empty((rows + 1) * cols, dtype=torch.int16, device="cuda"), ws)
    with pytest.raises(ValueError):
        afx.afx_prefill(d, dev, rows, cols, x, y, torch.empty(16, dtype=torch.int16, device="cuda"), ws)


@pytest.mark.slow
def test_prefill_qwen3_layer_matrices_sampled(afx):
    import torch
    n_tokens = 512
    rng = np.random.default_rng(0)
    for name, shape, kind in synth.LAYER_TENSORS:
        if kind != "matrix":
            continue
        rows, cols = shape
        W = synth.layer_tensor(name, seed=0)
        X = synth.activations(n_tokens, cols, seed=9)
        c, d = afx.encode(W.reshape(-1))
        y, scratch, ws = _bufs(afx, rows, cols, n_tokens)
        afx.afx_prefill(d, torch.from_numpy(c).cuda(), rows, cols, torch.from_numpy(X.view(np.int16)).cuda(), y,
                        scratch, ws)
        torch.cuda.synchronize()
        pick = rng.choice(rows, size=32, replace=False)
        ok, worst = _within(y.cpu().numpy()[:, pick], W[pick], X)
        assert ok, (name, worst)
