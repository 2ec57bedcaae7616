"""Host-side helpers of the bench's legs, on CPU: the comparison of the fused
product with restore-then-GEMM picks the fastest unfused form per batch and
skips batches that one of the two legs did not run; the host-encode leg
re-encodes the step's tensors and checks the containers are the same; the
committed traffic records name kernels and workloads that exist."""
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


def test_host_encode_leg_reproduces_the_step_containers():
    import numpy as np
    from weight_streaming_canonical_gb300 import afx, synth
    parts = []
    for seed, n in ((1, 70_000), (2, 5120)):
        w = synth.normal(n, seed=seed)
        c, d = afx.encode(w)
        parts.append((f"t{seed}", w, c, d))
    out = bench.run_host_encode(afx, parts, reps=1)
    assert out["containers_identical"]
    assert out["ms"] > 0 and out["weights_per_s"] > 0
    assert abs(out["input_gbs"] - 2 * 75_120 / (out["ms"] * 1e-3) / 1e9) < 1e-9
    # a container that differs from what the encoder writes is reported
    bad = list(parts)
    c2 = parts[0][2].copy()
    c2[-1] ^= 1
    bad[0] = (parts[0][0], parts[0][1], c2, parts[0][3])
    assert not bench.run_host_encode(afx, bad, reps=1)["containers_identical"]
    assert np.array_equal(parts[0][2], afx.encode(parts[0][1])[0])


def test_cpu_baseline_keeps_every_reported_thread_busy(monkeypatch):
    # 10 full slices and a short tensor for 4 threads: 8 slices, 2 a thread,
    # and the short tensor is not part of the sample
    from weight_streaming_canonical_gb300 import afx, synth
    monkeypatch.setattr(bench.os, "cpu_count", lambda: 4)
    parts = []
    for seed, n in ((1, 10 * bench.ORACLE_SLICE + 123), (2, 5120)):
        w = synth.normal(n, seed=seed)
        c, d = afx.encode(w)
        parts.append((f"t{seed}", w, c, d))
    out = bench.run_cpu_baseline(parts)
    assert out["cores"] == 4
    assert out["sample"].startswith("8 containers (16777216 weights)")
    assert "2 per thread on 4 threads" in out["sample"]
    assert out["one_core_weights_per_s"] > 0 and out["weights_per_s"] > 0
    # fewer slices than threads: one slice per busy thread, the rest not counted
    monkeypatch.setattr(bench.os, "cpu_count", lambda: 64)
    assert bench.run_cpu_baseline(parts)["cores"] == 10


def test_data_text_names_each_workloads_inputs():
    assert "Qwen3-14B layer shapes" in bench.data_text("layer")
    assert "NaN" in bench.data_text("adversarial")
    assert "4096x4096" in bench.data_text("matrix4096")
    assert "2^26" in bench.data_text("normal:26")
    assert all(bench.data_text(w).startswith("synthetic") for w in bench.WORKLOADS)


def test_every_traffic_record_names_a_kernel_and_a_workload():
    # profiles/<kernel>[.<workload>].traffic.json: the kernel is one the
    # sources define, the workload one the bench runs, the file name agrees
    # with the record, and the record's sources exist
    import glob
    import json
    import os
    import re
    recs = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.traffic.json")))
    assert recs
    src = open(os.path.join(bench.ROOT, "weight_streaming_canonical_gb300", "csrc", "afx_decode.cu")).read()
    kernels = set(re.findall(r"\b(restore_\w*kernel)\s*\(const __grid_constant__", src))
    assert "restore_store_pair_kernel" in kernels and "restore_store_kernel" in kernels
    for path in recs:
        rec = json.load(open(path))
        name = os.path.basename(path)[: -len(".traffic.json")]
        kernel, _, workload = name.partition(".")
        assert rec["kernel"] == kernel and kernel in kernels, path
        assert rec.get("bench_workload", "layer") == (workload or rec.get("bench_workload", "layer")), path
        assert rec.get("bench_workload", "layer") in bench.WORKLOADS, path
        assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"] > 0, path
        for s in rec["source"]:
            assert os.path.exists(os.path.join(bench.ROOT, s)), (path, s)
