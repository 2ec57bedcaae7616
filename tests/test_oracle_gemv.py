"""Pins for the oracle GEMV: closed forms and an independent float64 matmul."""
import numpy as np
import pytest

import oracle
from weight_streaming_canonical_gb300 import synth


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def test_unit_vector_selects_a_column_not_a_row():
    W = synth.normal(37 * 53, seed=4).reshape(37, 53)  # non-square: a transposed operand fails
    for j in (0, 7, 52):
        x = np.zeros((1, 53), np.uint16)
        x[0, j] = 0x3F80  # 1.0
        y, A = oracle.gemv(W, x)
        assert np.array_equal(y[0], _f(W[:, j]))
        assert np.array_equal(A[0], np.abs(_f(W[:, j]).astype(np.float64)))


def test_zero_input_gives_zero():
    W = synth.normal(64 * 96, seed=5).reshape(64, 96)
    y, A = oracle.gemv(W, np.zeros((3, 96), np.uint16))
    assert not y.any() and not A.any()


def test_all_ones_integer_sum_is_exact():
    W = np.full((5, 300), 0x3F80, np.uint16)  # 1.0 everywhere
    rng = np.random.default_rng(0)
    xi = rng.integers(-8, 9, size=(2, 300))
    x = synth.bf16_round(xi.astype(np.float32))
    y, A = oracle.gemv(W, x)
    assert np.array_equal(y, np.repeat(xi.sum(axis=1, keepdims=True), 5, axis=1).astype(np.float32))
    assert np.array_equal(A, np.repeat(np.abs(xi).sum(axis=1, keepdims=True), 5, axis=1).astype(np.float64))


@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_matches_float64_matmul(B):
    rows, cols = 129, 1031
    W = synth.normal(rows * cols, seed=6).reshape(rows, cols)
    x = synth.activations(B, cols, seed=7)
    y, A = oracle.gemv(W, x)
    Wf = _f(W).astype(np.float64)
    xf = _f(x).astype(np.float64)
    ref = xf @ Wf.T
    assert np.allclose(y, ref.astype(np.float32), rtol=1e-6, atol=1e-9)
    assert np.allclose(A, np.abs(xf[:, None, :] * Wf[None, :, :]).sum(-1), rtol=1e-12)
    # batches are independent: row b of x alone gives row b of y
    for b in range(B):
        yb, _ = oracle.gemv(W, x[b:b + 1])
        assert np.array_equal(yb[0], y[b])
