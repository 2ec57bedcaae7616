"""afx_plan_residency (host): exact against brute force on small instances,
the limiting budgets, Eq. (2)'s break-even between streaming the container
and streaming the BF16 weights, and feasibility at full model scale."""
import itertools

import numpy as np
import pytest

from weight_streaming_canonical_gb300 import synth


def _costs(S, C, link, restore, overlapped):
    """(resident bytes, ms) of the three placements the plan chooses among."""
    b, r = link * 1e6, restore * 1e6  # bytes per ms
    t_unpack = S / r
    stream_c = max(C / b, t_unpack) if overlapped else C / b + t_unpack
    return [(S, 0.0), (C, t_unpack), (0, min(stream_c, S / b))]


def _brute(tensors, budget, link, restore, overlapped):
    opts = [_costs(S, C, link, restore, overlapped) for S, C in tensors]
    best = None
    for pick in itertools.product(range(3), repeat=len(tensors)):
        mem = sum(opts[i][k][0] for i, k in enumerate(pick))
        if mem > budget:
            continue
        t = sum(opts[i][k][1] for i, k in enumerate(pick))
        best = t if best is None else min(best, t)
    return best


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("overlapped", [False, True])
def test_matches_brute_force(afx, seed, overlapped):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 7))
    tensors = []
    for _ in range(n):
        S = int(rng.integers(100, 5000)) * 2
        C = int(S * rng.uniform(0.5, 0.95))
        tensors.append((S, C))
    budget = int(rng.integers(0, sum(S for S, _ in tensors) + 1))  # < 65536 units: one byte per unit
    link, restore = float(rng.uniform(20, 400)), float(rng.uniform(50, 3000))
    place, ms, resident = afx.afx_plan_residency(tensors, budget, link, restore, overlapped)
    assert resident <= budget
    assert ms == pytest.approx(_brute(tensors, budget, link, restore, overlapped), rel=1e-12, abs=1e-15)
    # the reported time and bytes are those of the reported placements
    b, r = link * 1e6, restore * 1e6
    t, mem = 0.0, 0
    for (S, C), p in zip(tensors, place):
        if p == afx.AFX_RESIDENT_DECODED:
            mem += S
        elif p == afx.AFX_RESIDENT_COMPRESSED:
            mem += C
            t += S / r
        elif p == afx.AFX_STREAM_COMPRESSED:
            t += max(C / b, S / r) if overlapped else C / b + S / r
        else:
            assert p == afx.AFX_STREAM_RAW
            t += S / b
    assert mem == resident and t == pytest.approx(ms, rel=1e-12, abs=1e-15)


def test_enough_memory_keeps_everything_decoded(afx):
    tensors = [(2_000_000, 1_400_000), (10_000, 9_000), (6_000_000, 3_000_000)]
    place, ms, resident = afx.afx_plan_residency(tensors, 10**9, 200.0, 1000.0)
    assert place == [afx.AFX_RESIDENT_DECODED] * 3 and ms == 0.0 and resident == 8_010_000


@pytest.mark.parametrize("overlapped", [False, True])
def test_no_memory_streams_by_eq2(afx, overlapped):
    # Eq. (2) as written: the container pays when (S - C) / b > t_unpack
    S, C, b = 1_000_000, 650_000, 100.0
    saved_ms = (S - C) / (b * 1e6)
    for restore, expect in ((S / (0.5 * saved_ms) / 1e6, afx.AFX_STREAM_COMPRESSED),   # t_unpack = half the saving
                            (S / (2.0 * saved_ms) / 1e6, afx.AFX_STREAM_RAW)):         # twice the saving
        place, ms, resident = afx.afx_plan_residency([(S, C)], 0, b, restore, overlapped=False)
        assert place == [expect] and resident == 0
    # overlapped, the container wins whenever the restore is faster than the raw copy
    place, _, _ = afx.afx_plan_residency([(S, C)], 0, b, S / (0.9 * S / (b * 1e6)) / 1e6, overlapped=True)
    assert place == [afx.AFX_STREAM_COMPRESSED]


def test_compressed_residency_when_decoded_does_not_fit(afx):
    tensors = [(4_000, 2_600)]
    place, ms, resident = afx.afx_plan_residency(tensors, 3_000, 10.0, 1000.0)
    assert place == [afx.AFX_RESIDENT_COMPRESSED] and resident == 2_600


def test_qwen3_14b_model_plans_fit_and_improve_with_memory(afx):
    # the model's 362 tensors at N(0, 0.02) sizes (10.9 bits per weight), measured GB300 rates
    tensors = []
    for _ in range(synth.LAYERS):
        for name, shape, kind in synth.LAYER_TENSORS:
            n = synth.numel(shape)
            tensors.append((2 * n, int(n * (10.92 if kind == "matrix" else 9.1) / 8)))
    for shape in (synth.EMBED_SHAPE, synth.HEAD_SHAPE):
        n = synth.numel(shape)
        tensors.append((2 * n, int(n * 10.92 / 8)))
    assert len(tensors) == 362
    last = None
    for gb in (0, 8, 16, 24, 32, 48):
        place, ms, resident = afx.afx_plan_residency(tensors, gb << 30, 207.0, 2900.0)
        assert resident <= gb << 30
        assert last is None or ms <= last + 1e-9
        last = ms
    place, ms, resident = afx.afx_plan_residency(tensors, 30 << 30, 207.0, 2900.0)
    assert all(p == afx.AFX_RESIDENT_DECODED for p in place) and ms == 0.0  # 29.5 GB fits in 30 GiB


def test_bad_arguments(afx):
    with pytest.raises(afx.AfxError):
        afx.afx_plan_residency([], 100, 1.0, 1.0)
    with pytest.raises(afx.AfxError):
        afx.afx_plan_residency([(2, 1)], 100, 0.0, 1.0)
    with pytest.raises(afx.AfxError):
        afx.afx_plan_residency([(2, 1)], 100, 1.0, float("nan"))
