"""afx_decode_gemv_static: the fused restore + GEMV for callers that cannot
allocate device memory (it uses the library's own fixed device workspace).

Collected last on purpose.  Its results must match afx_decode_gemv, which
takes a caller-allocated workspace, on two calls in a row (the shared
workspace keeps the previous call's contents)."""
import ctypes

import numpy as np
import pytest

import oracle
from afx_testutil import within_gemv_tolerance
from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu


def _reference(afx, d, dev, rows, cols, xd):
    import torch
    B = xd.shape[0]
    y = torch.full((B, rows), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(afx.afx_decode_gemv_workspace(d, B) // 4 + 4, dtype=torch.float32, device="cuda")
    afx.afx_decode_gemv(d, dev, rows, cols, xd, y, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("shape,B", [((512, 5120), 4), ((3, 200_000), 2), ((1024, 72), 1)])
def test_static_workspace_matches_the_allocating_entry_point(afx, shape, B):
    import torch
    rows, cols = shape
    W = synth.normal(rows * cols, seed=rows).reshape(rows, cols)
    x = synth.activations(B, cols, seed=cols)
    c, d = afx.encode(W.reshape(-1))
    dev = torch.from_numpy(c).cuda()
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    y_ref = _reference(afx, d, dev, rows, cols, xd)
    y_oracle, A = oracle.gemv(W, x)
    assert within_gemv_tolerance(y_ref, y_oracle, A)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the second call finds the first call's partials in the workspace
        y = torch.full((B, rows), float("nan"), dtype=torch.float32, device="cuda")
        afx.afx_decode_gemv_static(d, dev, rows, cols, xd, y, status_dev=status)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert status.item() == 0
        assert within_gemv_tolerance(got, y_ref, A)
        assert within_gemv_tolerance(got, y_oracle, A)


def test_static_workspace_rejects_containers_that_need_more(afx):
    import torch
    w = synth.normal(5120 * 16, seed=1)
    code = afx.afx_build_code(w)
    factor = 1 << 16  # the same exponent mix at 5.4G weights: far more blocks than the static workspace covers
    for s in range(256):
        code.count[s] = code.count[s] * factor
    n = w.size * factor
    d = afx.afx_encode_bound(n, code)
    assert afx.afx_decode_gemv_workspace(d, 4) > afx.AFX_STATIC_WORKSPACE_BYTES
    dummy = torch.zeros(256, dtype=torch.uint8, device="cuda")
    x = torch.zeros((4, 5120), dtype=torch.int16, device="cuda")
    y = torch.zeros((4, n // 5120), dtype=torch.float32, device="cuda")
    with pytest.raises(afx.AfxError) as err:
        afx.afx_decode_gemv_static(d, dummy, n // 5120, 5120, x, y)
    assert err.value.status == afx.AFX_E_NOSPACE
    assert "static workspace" in str(err.value)
