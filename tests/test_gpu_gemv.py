"""Fused decode + GEMV parity: afx_decode_gemv (through the C ABI) against the
oracle GEMV on the oracle-decoded weights, |err| <= 2e-3 * sum|w x| per
output, plus closed forms and run-to-run reproducibility."""
import numpy as np
import pytest

import oracle
from afx_testutil import gpu_gemv, within_gemv_tolerance
from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu


def _check(afx, W, x):
    rows, cols = W.shape
    c, d = afx.encode(W.reshape(-1))
    Wd, st = oracle.decode(c)
    assert st == oracle.OK
    y_ref, A = oracle.gemv(Wd.reshape(rows, cols), x)
    y, status = gpu_gemv(afx, c, d, rows, cols, x)
    assert status == 0
    assert not np.isnan(y).any(), "an output was never written"
    assert within_gemv_tolerance(y, y_ref, A), float(np.max(np.abs(y - y_ref) / np.maximum(A, 1e-30)))
    return y, c, d


SHAPES = [(64, 64), (3, 5120), (257, 1000), (100, 5120), (7, 17408), (1024, 72), (41, 4099), (2000, 128)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_shapes_and_batches(afx, shape, B):
    rows, cols = shape
    W = synth.normal(rows * cols, seed=rows + cols).reshape(rows, cols)
    x = synth.activations(B, cols, seed=B)
    _check(afx, W, x)


@pytest.mark.parametrize("cols", [2056, 2064, 2072])
def test_rows_at_the_warp_path_boundary(afx, cols):
    # 2064 columns and more (a multiple of 8): one warp's run of 32 chunks meets at most two rows
    W = synth.normal(500 * cols, seed=cols).reshape(500, cols)
    x = synth.activations(4, cols, seed=cols)
    _check(afx, W, x)


def test_corrupt_stream_is_flagged_by_the_gemv(afx):
    import torch
    rows, cols = 200, 5120
    W = synth.normal(rows * cols, seed=21).reshape(rows, cols)
    c, d = afx.encode(W.reshape(-1))
    bad = c.copy()
    rng = np.random.default_rng(2)
    bad[d.off_exp: d.off_exp + d.n_chunks * d.chunk_bytes] = rng.integers(
        0, 256, size=d.n_chunks * d.chunk_bytes, dtype=np.uint8)
    y, status = gpu_gemv(afx, bad, d, rows, cols, synth.activations(2, cols, seed=5))
    assert status != 0


def test_unit_vector_gives_a_column_exactly(afx):
    rows, cols = 300, 5120
    W = synth.normal(rows * cols, seed=1).reshape(rows, cols)
    for j in (0, 4095, 5119):
        x = np.zeros((1, cols), np.uint16)
        x[0, j] = 0x3F80
        c, d = afx.encode(W.reshape(-1))
        y, status = gpu_gemv(afx, c, d, rows, cols, x)
        assert status == 0
        col = (W[:, j].astype(np.uint32) << 16).view(np.float32)
        assert np.array_equal(y[0], col)


@pytest.mark.parametrize("B", [2, 3, 4])
def test_unit_vector_per_batch_row_gives_its_own_column_exactly(afx, B):
    # batch row b selects column j_b: every (row, batch) sum has one nonzero
    # product, so y[b] is W[:, j_b] exactly and a sum sent to the wrong
    # (row, batch) slot by the reduction shows up as a wrong column
    rows, cols = 300, 5120
    W = synth.normal(rows * cols, seed=6).reshape(rows, cols)
    js = [0, 5119, 2500, 4095][:B]
    x = np.zeros((B, cols), np.uint16)
    for b, j in enumerate(js):
        x[b, j] = 0x3F80
    c, d = afx.encode(W.reshape(-1))
    y, status = gpu_gemv(afx, c, d, rows, cols, x)
    assert status == 0
    for b, j in enumerate(js):
        assert np.array_equal(y[b], (W[:, j].astype(np.uint32) << 16).view(np.float32)), (b, j)


def test_zero_activation_gives_zero(afx):
    W = synth.normal(64 * 5120, seed=2).reshape(64, 5120)
    c, d = afx.encode(W.reshape(-1))
    y, status = gpu_gemv(afx, c, d, 64, 5120, np.zeros((4, 5120), np.uint16))
    assert status == 0 and not y.any()


def test_reproducible_bit_for_bit(afx):
    W = synth.normal(333 * 5120, seed=3).reshape(333, 5120)
    x = synth.activations(4, 5120, seed=3)
    c, d = afx.encode(W.reshape(-1))
    y1, _ = gpu_gemv(afx, c, d, 333, 5120, x)
    y2, _ = gpu_gemv(afx, c, d, 333, 5120, x)
    assert np.array_equal(y1, y2)


def test_row_longer_than_a_block(afx):
    # one row spans several decode blocks: the fix-up pass joins the partials
    W = synth.normal(3 * 200_000, seed=4).reshape(3, 200_000)
    x = synth.activations(2, 200_000, seed=4)
    _check(afx, W, x)


def test_single_exponent_matrix(afx):
    W = (np.full((50, 640), 0x3F80, np.uint16) | (np.arange(50 * 640).reshape(50, 640) % 128).astype(np.uint16))
    _check(afx, W, synth.activations(3, 640, seed=5))


def test_bad_arguments(afx):
    import torch
    W = synth.normal(64 * 128, seed=6).reshape(64, 128)
    c, d = afx.encode(W.reshape(-1))
    dev = torch.from_numpy(c).cuda()
    x = torch.zeros((5, 128), dtype=torch.int16, device="cuda")
    y = torch.zeros((5, 64), dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 16, dtype=torch.float32, device="cuda")
    with pytest.raises(afx.AfxError):
        afx.afx_decode_gemv(d, dev, 64, 128, x, y, ws)  # batch 5
    with pytest.raises(afx.AfxError):
        afx.afx_decode_gemv(d, dev, 32, 128, x[:1], y, ws)  # rows * cols != n
    with pytest.raises(afx.AfxError):
        afx.afx_decode_gemv(d, dev, 64, 128, x[:1], y, ws[:1])  # workspace too small


@pytest.mark.slow
@pytest.mark.parametrize("B", [1, 4])
def test_qwen3_layer_matrices(afx, B):
    for name, shape, kind in synth.LAYER_TENSORS:
        if kind != "matrix":
            continue
        W = synth.layer_tensor(name, seed=0)
        x = synth.activations(B, shape[1], seed=10 + B)
        _check(afx, W, x)


def test_gemv_batch_of_products_in_one_launch(afx):
    import torch
    shapes = [(96, 640), (640, 1024), (33, 5120), (1024, 72), (3, 200_000)]
    B = 3
    items = []
    for i, (r, c) in enumerate(shapes):
        W = synth.normal(r * c, seed=200 + i).reshape(r, c)
        x = synth.activations(B, c, seed=300 + i)
        cont, d = afx.encode(W.reshape(-1))
        items.append((W, x, cont, d))
    devs = [torch.from_numpy(cont).cuda() for _, _, cont, _ in items]
    xs = [torch.from_numpy(x.view(np.int16)).cuda() for _, x, _, _ in items]
    ys = [torch.full((B, r), float("nan"), dtype=torch.float32, device="cuda") for r, _ in shapes]
    wss = [torch.empty(afx.afx_decode_gemv_workspace(d, B) // 4 + 4, dtype=torch.float32, device="cuda")
           for _, _, _, d in items]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_gemv_batch([d for *_, d in items], devs, shapes, xs, ys, wss, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for (W, x, _, _), y in zip(items, ys):
        y_ref, A = oracle.gemv(W, x)
        assert within_gemv_tolerance(y.cpu().numpy(), y_ref, A)


@pytest.mark.parametrize("B", [1, 2, 4])
def test_partial_state_table(afx, B):
    # 90 exponents: rows for the shallowest 50 internal nodes of 89, escapes
    # at the others (launches of their own)
    rows, cols = 300, 5120
    W = synth.exponent_mix(rows * cols, 90, ratio=0.9, seed=B).reshape(rows, cols)
    x = synth.activations(B, cols, seed=B)
    _, _, d = _check(afx, W, x)
    assert d.nsym == 90 and afx.afx_decode_table_kind(d)[0] == afx.AFX_TABLE_PARTIAL


def test_gemv_batch_mixing_partial_and_whole_state_tables(afx):
    import torch
    shapes = [(200, 5120), (150, 2560), (64, 17408), (96, 640)]
    B = 4
    items = []
    for i, (r, c) in enumerate(shapes):
        if i % 2:  # 90 exponents (a partial state table) and 130 (the 12-bit table)
            W = synth.exponent_mix(r * c, 70 + 20 * i, ratio=0.9, seed=400 + i).reshape(r, c)
        else:
            W = synth.normal(r * c, seed=400 + i).reshape(r, c)
        x = synth.activations(B, c, seed=500 + i)
        cont, d = afx.encode(W.reshape(-1))
        items.append((W, x, cont, d))
    devs = [torch.from_numpy(cont).cuda() for _, _, cont, _ in items]
    xs = [torch.from_numpy(x.view(np.int16)).cuda() for _, x, _, _ in items]
    ys = [torch.full((B, r), float("nan"), dtype=torch.float32, device="cuda") for r, _ in shapes]
    wss = [torch.empty(afx.afx_decode_gemv_workspace(d, B) // 4 + 4, dtype=torch.float32, device="cuda")
           for _, _, _, d in items]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_gemv_batch([d for *_, d in items], devs, shapes, xs, ys, wss, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for (W, x, _, _), y in zip(items, ys):
        y_ref, A = oracle.gemv(W, x)
        assert within_gemv_tolerance(y.cpu().numpy(), y_ref, A)
