"""The bench's multi-rank host logic on CPU: two gloo ranks, the barrier, the
max over ranks of the step time, the whole-job throughput, and the
reference arm running on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out) -> None:
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = bench.max_over_ranks(1.0 + 2.0 * rank, world)  # rank 1 is the slow one
        value, wps = bench.job_throughput(1_000_000, world, ms)
        bench.barrier(world)
        out.put((rank, ms, value, wps))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value, wps in got:
        assert ms == 3.0  # the max over ranks
        assert wps == pytest.approx(2 * 1_000_000 / 3e-3)
        assert value == pytest.approx(2 * 2 * 1_000_000 / 3e-3 / 1e9)


def test_job_throughput_is_weak_scaling():
    v1, w1 = bench.job_throughput(330_311_680, 1, 0.25)
    v8, w8 = bench.job_throughput(330_311_680, 8, 0.25)
    assert v8 == pytest.approx(8 * v1) and w8 == pytest.approx(8 * w1)
    assert v1 == pytest.approx(2 * 330_311_680 / 0.25e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    bench.run_reference(args)  # rank 1 returns at once, printing nothing
    assert capsys.readouterr().out == ""


def test_reference_arm_loads_only_the_oracle():
    # the reference arm encodes its sample with the oracle itself: run it in
    # a fresh process and check which shared objects of this repository it mapped
    code = (
        "import json, sys, bench\n"
        "bench.run_reference(bench.parse_args(['--impl', 'reference', '--workload', 'normal:21', "
        "'--steps', '1', '--warmup', '3']))\n"
        "maps = open('/proc/self/maps').read()\n"
        "print(json.dumps({'afx': 'libafx' in maps, 'orc': 'liborc' in maps}))\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=300,
                         env={**os.environ, "WORLD_SIZE": "1", "RANK": "0"})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [json.loads(x) for x in out.stdout.splitlines() if x.startswith("{")]
    ref, maps = lines[0], lines[-1]
    assert ref["impl"] == "reference" and ref["value"] > 0
    assert ref["config"]["weights_per_step"] == 1 << 21
    assert maps == {"afx": False, "orc": True}
