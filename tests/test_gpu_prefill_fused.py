"""The fused restore + tensor-core product for prefill (afx_prefill_fused,
afx_prefill_fused_batch): weights encoded in tile order, restored inside
the product, every output checked against the oracle's GEMV (float64
products and sums of the original row-major BF16 weights, one token vector
per batch row), |err| <= 2e-3 * sum|w x| per output."""
import numpy as np
import pytest

import oracle
from afx_testutil import within_gemv_tolerance
from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu


def _within(y, W, X):
    y_ref, A = oracle.gemv(np.ascontiguousarray(W), np.ascontiguousarray(X))
    err = np.abs(y.astype(np.float64) - y_ref.astype(np.float64))
    return within_gemv_tolerance(y, y_ref, A), float(np.max(err / np.maximum(A, 1e-30)))


def _tiled(afx, W):
    rows, cols = W.shape
    return afx.encode(afx.afx_tile_order(W, rows, cols))


def _workspace(afx, rings=None):
    import torch
    n = afx.afx_prefill_fused_workspace() if rings is None else rings * 16 * 16384
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def _run(afx, W, X, status=None, ws=None):
    import torch
    rows, cols = W.shape
    c, d = _tiled(afx, W)
    y = torch.full((X.shape[0], rows), float("nan"), dtype=torch.float32, device="cuda")
    afx.afx_prefill_fused(d, torch.from_numpy(c).cuda(), rows, cols, torch.from_numpy(X.view(np.int16)).cuda(), y,
                          _workspace(afx) if ws is None else ws, status_dev=status)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("shape", [(128, 64), (256, 640), (384, 5120), (1024, 192)])
@pytest.mark.parametrize("n_tokens", [1, 17, 128, 300, 512])
def test_fused_prefill_matches_the_oracle(afx, shape, n_tokens):
    import torch
    rows, cols = shape
    W = synth.normal(rows * cols, seed=rows + n_tokens).reshape(rows, cols)
    X = synth.activations(n_tokens, cols, seed=cols + 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = _run(afx, W, X, status)
    assert status.item() == 0
    ok, worst = _within(y, W, X)
    assert ok, worst


@pytest.mark.parametrize("n_tokens", [513, 1100, 2048])
def test_fused_prefill_several_passes(afx, n_tokens):
    # more than 512 tokens: the weights are restored once per pass of 512
    rows, cols = 256, 1024
    W = synth.normal(rows * cols, seed=n_tokens).reshape(rows, cols)
    X = synth.activations(n_tokens, cols, seed=3)
    ok, worst = _within(_run(afx, W, X), W, X)
    assert ok, worst


def test_fused_prefill_closed_forms(afx):
    # x = e_j selects column j of W exactly; x = 0 gives 0; all-ones W with
    # small-integer x gives exact integer sums
    rows, cols = 128, 192
    W = synth.normal(rows * cols, seed=5).reshape(rows, cols)
    X = np.zeros((3, cols), dtype=np.uint16)
    X[0, 7] = 0x3F80   # 1.0
    X[1, 130] = 0x3F80
    y = _run(afx, W, X)
    f = (W.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(y[0], f[:, 7]) and np.array_equal(y[1], f[:, 130])
    assert np.all(y[2] == 0)
    ones = np.full((rows, cols), 0x3F80, dtype=np.uint16)
    xi = np.arange(cols, dtype=np.float32) % 5 - 2
    Xi = (xi.view(np.uint32) >> 16).astype(np.uint16).reshape(1, cols)
    y1 = _run(afx, ones, Xi)
    assert np.all(y1 == xi.sum())


def test_fused_prefill_is_reproducible(afx):
    import torch
    rows, cols, n_tokens = 512, 2048, 200
    W = synth.normal(rows * cols, seed=9).reshape(rows, cols)
    X = synth.activations(n_tokens, cols, seed=10)
    c, d = _tiled(afx, W)
    dev = torch.from_numpy(c).cuda()
    xd = torch.from_numpy(X.view(np.int16)).cuda()
    outs = []
    ws = _workspace(afx)
    for _ in range(3):
        y = torch.empty((n_tokens, rows), dtype=torch.float32, device="cuda")
        afx.afx_prefill_fused(d, dev, rows, cols, xd, y, ws)
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy())
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])


def test_fused_prefill_batch_mixed_matrices(afx):
    # several matrices of different widths in one launch, one of them with a
    # single exponent for every weight (no coded stream: a fill)
    import torch
    shapes = [(256, 1024), (128, 5120), (640, 640), (128, 192), (384, 2048)]
    n_tokens = 96
    items = []
    for i, (r, cl) in enumerate(shapes):
        if i == 3:
            rng = np.random.default_rng(1)
            W = ((np.uint16(121) << 7) | rng.integers(0, 128, size=r * cl).astype(np.uint16)
                 | (rng.integers(0, 2, size=r * cl).astype(np.uint16) << 15)).reshape(r, cl)
        else:
            W = synth.normal(r * cl, seed=800 + i).reshape(r, cl)
        X = synth.activations(n_tokens, cl, seed=900 + i)
        c, d = _tiled(afx, W)
        items.append((W, X, torch.from_numpy(c).cuda(), d, torch.from_numpy(X.view(np.int16)).cuda()))
    assert items[3][3].nsym == 1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = _workspace(afx)
    for _ in range(2):  # the second call finds the first call's tiles in the workspace
        ys = [torch.full((n_tokens, r), float("nan"), dtype=torch.float32, device="cuda") for r, _ in shapes]
        afx.afx_prefill_fused_batch([it[3] for it in items], [it[2] for it in items], shapes,
                                    [it[4] for it in items], ys, ws, status_dev=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        for (W, X, *_), y in zip(items, ys):
            ok, worst = _within(y.cpu().numpy(), W, X)
            assert ok, worst


@pytest.mark.parametrize("n_exponents", [40, 60])
def test_fused_prefill_large_code_trees_use_the_12_bit_table(afx, n_exponents):
    # code trees with more internal nodes than the fused kernel's state table
    # holds (40 exponents: the restore kernel's state table would hold it; 60:
    # past every state table)
    rows, cols, n_tokens = 256, 4096, 64
    W = synth.exponent_mix(rows * cols, n_exponents, seed=n_exponents).reshape(rows, cols)
    X = synth.activations(n_tokens, cols, seed=4)
    c, d = _tiled(afx, W)
    assert d.nsym == n_exponents
    ok, worst = _within(_run(afx, W, X), W, X)
    assert ok, worst


@pytest.mark.parametrize("rings", [1, 3])
def test_fused_prefill_with_a_small_workspace(afx, rings):
    # a workspace of one or three rings runs that many CTAs over all the items
    rows, cols, n_tokens = 1024, 640, 100
    W = synth.normal(rows * cols, seed=rings).reshape(rows, cols)
    X = synth.activations(n_tokens, cols, seed=7)
    ok, worst = _within(_run(afx, W, X, ws=_workspace(afx, rings)), W, X)
    assert ok, worst


def test_fused_prefill_refuses_bad_arguments(afx):
    import torch
    W = synth.normal(128 * 64, seed=1).reshape(128, 64)
    c, d = _tiled(afx, W)
    dev = torch.from_numpy(c).cuda()
    x = torch.zeros((4, 64), dtype=torch.int16, device="cuda")
    y = torch.zeros((4, 128), dtype=torch.float32, device="cuda")
    ws = _workspace(afx, 1)
    with pytest.raises(afx.AfxError):  # rows not a multiple of 128
        afx.afx_prefill_fused(d, dev, 64, 128, torch.zeros((4, 128), dtype=torch.int16, device="cuda"),
                              torch.zeros((4, 64), dtype=torch.float32, device="cuda"), ws)
    with pytest.raises(afx.AfxError):  # cols not a multiple of 64
        afx.afx_prefill_fused(d, dev, 256, 32, torch.zeros((4, 32), dtype=torch.int16, device="cuda"),
                              torch.zeros((4, 256), dtype=torch.float32, device="cuda"), ws)
    with pytest.raises((afx.AfxError, ValueError)):  # x in host memory
        afx.afx_prefill_fused(d, dev, 128, 64, torch.zeros((4, 64), dtype=torch.int16), y, ws)
    c2, d2 = afx.encode(synth.normal_fp16(128 * 64, seed=2), fmt=afx.AFX_FMT_FP16)
    with pytest.raises(afx.AfxError):  # FP16 elements
        afx.afx_prefill_fused(d2, torch.from_numpy(c2).cuda(), 128, 64, x, y, ws)
    with pytest.raises(afx.AfxError) as err:  # a workspace smaller than one ring
        afx.afx_prefill_fused(d, dev, 128, 64, x, y, ws[: 16 * 16384 - 256])
    assert err.value.status == afx.AFX_E_NOSPACE
    afx.afx_prefill_fused(d, dev, 128, 64, x, y, ws)  # the same call with valid arguments
    torch.cuda.synchronize()


@pytest.mark.slow
@pytest.mark.parametrize("n_tokens", [512, 2048])
def test_fused_prefill_qwen3_layer_matrices_sampled(afx, n_tokens):
    # the layer's seven matrices in one batch call; 32 sampled rows of every
    # product against the oracle's GEMV of those rows
    import torch
    rng = np.random.default_rng(n_tokens)
    mats = [(name, shape) for name, shape, kind in synth.LAYER_TENSORS if kind == "matrix"]
    items = []
    for name, (rows, cols) in mats:
        W = synth.layer_tensor(name, seed=0)
        X = synth.activations(n_tokens, cols, seed=9)
        c, d = _tiled(afx, W)
        items.append((W, X, torch.from_numpy(c).cuda(), d, torch.from_numpy(X.view(np.int16)).cuda()))
    ys = [torch.full((n_tokens, r), float("nan"), dtype=torch.float32, device="cuda") for _, (r, _) in mats]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_prefill_fused_batch([it[3] for it in items], [it[2] for it in items], [s for _, s in mats],
                                [it[4] for it in items], ys, _workspace(afx), status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for (name, (rows, cols)), (W, X, *_), y in zip(mats, items, ys):
        pick = np.sort(rng.choice(rows, size=32, replace=False))
        ok, worst = _within(y.cpu().numpy()[:, pick], W[pick], X)
        assert ok, (name, worst)
