"""Host-side helpers of the bench's legs, on CPU: the comparison of the fused
product with restore-then-GEMM picks the fastest unfused form per batch and
skips batches that one of the two legs did not run."""
import bench


def test_fused_vs_unfused_takes_the_fastest_unfused_form():
    fused = {"batch1": {"ms": 0.25}, "batch4": {"ms": 0.35}}
    prefill = {"weights": 10, "runs": [
        {"tokens": 1, "sequential_ms": 0.45, "overlapped_ms": 0.44, "one_restore_launch_ms": 0.36},
        {"tokens": 4, "sequential_ms": 0.45, "overlapped_ms": 0.30, "one_restore_launch_ms": 0.36},
        {"tokens": 128, "sequential_ms": 0.5, "overlapped_ms": 0.5, "one_restore_launch_ms": 0.4}]}
    out = bench.fused_vs_unfused(fused, prefill)
    assert set(out) == {"batch1", "batch4"}
    assert out["batch1"]["unfused_form"] == "one_restore_launch"
    assert out["batch1"]["restore_then_gemm_ms"] == 0.36
    assert abs(out["batch1"]["unfused_over_fused"] - 0.36 / 0.25) < 1e-12
    assert out["batch4"]["unfused_form"] == "overlapped"
    assert abs(out["batch4"]["unfused_over_fused"] - 0.30 / 0.35) < 1e-12


def test_fused_vs_unfused_skips_missing_batches():
    out = bench.fused_vs_unfused({"batch1": {"ms": 0.25}}, {"weights": 1, "runs": [
        {"tokens": 4, "sequential_ms": 1.0, "overlapped_ms": 1.0, "one_restore_launch_ms": 1.0}]})
    assert out == {}
    assert bench.fused_vs_unfused({}, {"runs": []}) == {}
