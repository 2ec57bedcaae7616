#!/usr/bin/env python
"""Benchmark of the lossless BF16 weight restore (afx) on GB300.

One step restores every tensor of the whole Qwen3-14B-shaped model (40
decoder layers of q/k/v/o, gate/up/down and two norm vectors, plus the
embedding and the untied LM head: 14,768,291,840 BF16 weights, 29.5 GB)
from containers already resident in HBM, through the C ABI (one
afx_decode_batch call, captured once in a CUDA graph and replayed).
`--workload` picks another workload for the headline.

Reported: decoded BF16 GB/s (2 bytes x weights / step time) as `value`,
weights/s, HBM GB/s (compressed bytes read + BF16 bytes written) against
the measured copy bandwidth, the roofline of the restore kernel, an
end-to-end number through the C ABI from pinned host containers to a host
BF16 result, the CPU oracle on the host cores, and (`per_config`) the
4096x4096 matrix, the single layer and the 2^28 adversarial tensor, each
checked bit for bit before it is timed.  The layer's further legs (fused
GEMV, prefill, 40 streamed layers, formats, zero-copy, host encode)
follow.

`--impl reference` times the CPU oracle itself (the reference arm): the
bit-serial decoder on containers the oracle encodes itself, on the host
cores.

The decode is the t_unpack term of "Why Weight Offloading Slows
Inference", Eq. (1); the break-even it must meet is that page's Eq. (2).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decoded BF16 GB/s (and weights/s) per GB300; % of HBM roofline"
WORKLOAD = "qwen3-14b-shaped decoder layer: q,o 5120x5120; k,v 1024x5120; gate,up 17408x5120; down 5120x17408; 2 norms 5120"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20  # GB300 L2
BUSY_PAD_S = 0.5  # seconds of untimed identical steps on each side of the timed ones


def busy_pad_steps(step_ms: float) -> int:
    """Steps that fill about BUSY_PAD_S of GPU time (at least 1, at most 20000)."""
    if not step_ms > 0:
        return 1
    return max(1, min(20000, int(BUSY_PAD_S * 1e3 / step_ms + 0.5)))


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-extras", action="store_true",
                   help="the headline restore only: skip every leg after it (see --legs)")
    p.add_argument("--e2e-piece-weights", type=int, default=0,
                   help="end-to-end leg: store each tensor as containers of at most this many weights "
                        "(consecutive slices), streamed one per stage; 0: one container per tensor")
    p.add_argument("--config", type=int, choices=[1, 2, 3, 4, 5], default=None,
                   help="the five workloads by number: 1 the 4096x4096 matrix, 2 the layer, 3 the whole model, "
                        "4 the 2^28 adversarial tensor, 5 the layer with the 40-layer streaming leg")
    p.add_argument("--legs", default="all",
                   help="extra legs to run after the headline (comma list of e2e, zero_copy, cpu_baseline, configs, "
                        "gemv, stream, prefill, formats, encode, wide_trees; default all)")
    p.add_argument("--workload", default="model",
                   help="model (default: the whole Qwen3-14B-shaped model, 14.77 B weights resident), layer (one "
                        "Qwen3-14B-shaped decoder layer), matrix4096, normal:<k> (one "
                        "N(0,0.02) tensor of 2^k weights), adversarial "
                        "(2^28 heavy-tailed), tensor:<name> (one tensor of the layer), layer-fp16 or layer-e4m3 "
                        "(the layer in the other element formats)")
    args = p.parse_args(argv)
    if args.config is not None:
        args.workload = {1: "matrix4096", 2: "layer", 3: "model", 4: "adversarial", 5: "layer"}[args.config]
        if args.config == 5:
            args.legs = "stream"
    return args


# ---- distributed plumbing (barrier and max over ranks only) ----------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(weights_per_rank: int, world: int, ms_max: float, elem_bytes: int = 2) -> tuple[float, float]:
    """Whole-job decoded GB/s and weights/s: every rank restores its own
    copy of the workload (weak scaling); the slowest rank's time counts."""
    total = weights_per_rank * world
    sec = ms_max * 1e-3
    return elem_bytes * total / sec / 1e9, total / sec


# ---- workload ------------------------------------------------------------------------

WORKLOADS = {
    "layer": WORKLOAD,
    "model": "full qwen3-14b-shaped model: 40 layers + embedding and untied LM head 151936x5120, 14.77B BF16 weights",
    "matrix4096": "single 4096x4096 BF16 matrix, N(0,0.02)",
    "adversarial": "2^28 BF16: Student-t(3)*0.01, 1% x100, 5% zeros, subnormals, +-inf, NaN payloads",
    "layer-fp16": "the qwen3-14b-shaped decoder layer stored as FP16 (same shapes and distributions)",
    "layer-e4m3": "the qwen3-14b-shaped decoder layer's seven matrices stored as E4M3 with a per-tensor scale",
}

FMT_OF_WORKLOAD = {"layer-fp16": 1, "layer-e4m3": 2}


def fmt_of(parts) -> int:
    return int(parts[0][3].format) if parts else 0


def elem_bytes(fmt: int) -> int:
    return 1 if fmt == 2 else 2


def torch_elem_dtype(fmt: int):
    import torch
    return torch.uint8 if fmt == 2 else torch.int16


def np_elem_dtype(fmt: int):
    return np.uint8 if fmt == 2 else np.uint16


def workload_generators(seed: int, rank: int = 0, workload: str = "model"):
    """The workload's tensors in order, as {name: () -> element patterns}
    (nothing is generated until a generator is called)."""
    from weight_streaming_canonical_gb300 import synth

    if workload == "matrix4096":
        gens = {"matrix4096": lambda: synth.matrix_4096(seed=seed + rank)}
    elif workload == "adversarial":
        gens = {"adversarial": lambda: synth.adversarial(1 << 28, seed=seed + rank)}
    elif workload.startswith("tensor:"):
        name = workload.split(":", 1)[1]
        gens = {name: lambda: synth.layer_tensor(name, seed=seed, layer=rank)}
    elif workload.startswith("normal:"):
        lg = int(workload.split(":", 1)[1])
        if not 0 <= lg <= 30:
            raise SystemExit("normal:<k> takes 0 <= k <= 30")
        gens = {workload: lambda: synth.normal(1 << lg, seed=seed + lg + rank)}
    elif workload == "layer":
        gens = {name: (lambda nm=name: synth.layer_tensor(nm, seed=seed, layer=rank))
                for name, _, _ in synth.LAYER_TENSORS}
    elif workload == "layer-fp16":
        gens = {name: (lambda nm=name: synth.layer_tensor_fp16(nm, seed=seed, layer=rank))
                for name, _, _ in synth.LAYER_TENSORS}
    elif workload == "layer-e4m3":
        gens = {name: (lambda nm=name: synth.layer_matrix_e4m3(nm, seed=seed, layer=rank))
                for name, _, kind in synth.LAYER_TENSORS if kind == "matrix"}
    elif workload == "model":
        gens = {"embed_tokens": lambda: synth.embedding(seed=seed + rank)}
        for layer_index in range(synth.LAYERS):
            for name, _, _ in synth.LAYER_TENSORS:
                gens[f"layers.{layer_index}.{name}"] = (
                    lambda nm=name, li=layer_index: synth.layer_tensor(nm, seed=seed + rank, layer=li))
        gens["lm_head"] = lambda: synth.lm_head(seed=seed + rank)
    else:
        raise SystemExit(f"unknown workload {workload}")
    return gens


def build_layer(seed: int, rank: int = 0, workload: str = "model"):
    """Generate and encode the workload on the host: [(name, w, container, desc)]."""
    from weight_streaming_canonical_gb300 import afx

    gens = workload_generators(seed, rank, workload)
    fmt = FMT_OF_WORKLOAD.get(workload, 0)

    def one(item):
        name, gen = item
        w = np.ascontiguousarray(gen()).reshape(-1)
        c, d = afx.encode(w, fmt=fmt)
        return name, w, c, d

    with cf.ThreadPoolExecutor(min(len(gens), 16)) as ex:
        return list(ex.map(one, gens.items()))


def data_text(workload: str) -> str:
    """What the synthetic inputs are, for the JSON line's `data`."""
    fixed = {
        "layer": "synthetic: seeded N(0,0.02) BF16 matrices, N(1,0.05) norms, Qwen3-14B layer shapes",
        "model": "synthetic: seeded N(0,0.02) BF16 matrices, N(1,0.05) norms, Qwen3-14B model shapes",
        "layer-fp16": "synthetic: seeded N(0,0.02) matrices, N(1,0.05) norms rounded to FP16, Qwen3-14B layer shapes",
        "layer-e4m3": "synthetic: seeded N(0,1) x 448/6 matrices rounded to E4M3, Qwen3-14B layer matrix shapes",
        "adversarial": "synthetic: seeded heavy-tailed BF16 with zeros, subnormals, infinities and NaN payloads",
    }
    return fixed.get(workload, "synthetic: seeded " + workload_text(workload))


def workload_text(workload: str) -> str:
    if workload.startswith("tensor:"):
        return f"one tensor of the Qwen3-14B-shaped layer: {workload.split(':', 1)[1]}"
    if workload.startswith("normal:"):
        return f"one BF16 tensor of 2^{workload.split(':', 1)[1]} weights, N(0,0.02)"
    return WORKLOADS[workload]


def exponent_entropy_bits(parts) -> float:
    """Empirical entropy of the BF16 exponents per weight, weighted over the
    tensors (each tensor has its own code): the least any exponent code can
    spend, before the chunk and block index."""
    total, n_all = 0.0, 0
    for _, w, _, d in parts:
        sym = ((w.reshape(-1) >> 3) & 0xF if d.format == 2 else (w.reshape(-1) >> 10) & 0x1F if d.format == 1
               else (w.reshape(-1) >> 7) & 0xFF)
        counts = np.bincount(sym.astype(np.intp), minlength=256).astype(np.float64)
        p = counts[counts > 0] / w.size
        total += float(-(p * np.log2(p)).sum()) * w.size
        n_all += w.size
    return total / max(n_all, 1)


def algorithmic_bytes(d) -> int:
    """Bytes a restore must move: coded symbol bits, the raw bits (a sign|mantissa
    byte per element, plus FP16's 3 leading fraction bits; a nibble for E4M3),
    chunk and block index entries read; the elements written (2 bytes each; 1
    for E4M3).  FP16's hi section holds the 3 bits in a nibble: its fourth
    bit is the format's padding and is not counted, so the FP16 fraction
    errs low."""
    fmt = getattr(d, "format", 0)
    raw, out = ((d.n + 1) // 2, d.n) if fmt == 2 else (d.n, 2 * d.n)
    if fmt == 1:
        raw += (3 * d.n + 7) // 8  # FP16's hi section
    return (d.total_bits + 7) // 8 + raw + 2 * d.n_chunks + 8 * (d.n_blocks + 1) + out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms with the
    sample's wall-clock time.  stop(window) keeps the samples taken inside the
    host-time window (t0, t1) during which the GPU was kept busy around the
    timed steps."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    @staticmethod
    def _wall(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    @classmethod
    def summarize(cls, lines, window=None):
        """Median SM clock, highest max clock, median power and the throttle
        reasons seen, over the samples inside window (all samples when none
        falls inside it or no window is given)."""
        rows = []
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            try:
                watts = float(f[3])
            except ValueError:
                watts = None
            active = {name for name, val in zip(cls.REASONS, f[5:9]) if val.lower() == "active"}
            rows.append((cls._wall(f[0]), sm, mx, watts, active))
        if not rows:
            return None
        inside = rows
        if window is not None:
            t0, t1 = window
            inside = [r for r in rows if r[0] is not None and t0 <= r[0] <= t1]
        scope = "samples taken while the GPU ran the timed steps and the same work around them"
        if not inside:
            inside, scope = rows, "no sample fell inside the busy window: all samples of the run"
        watts = [r[3] for r in inside if r[3] is not None]
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(set().union(*(r[4] for r in inside))), "samples": len(inside),
                "power_w": statistics.median(watts) if watts else None, "scope": scope}

    def stop(self, window=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarize(out.splitlines(), window)


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu capture of `kernel` on
    this workload (profiles/<kernel>.<workload>.traffic.json, else the
    kernel's main record), or None when no capture is of this workload or
    the kernel source has changed since (the sha256 of the source files,
    concatenated in the record's order, is stored with the counters)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}.{workload}.traffic.json")
    if not os.path.exists(path):
        path = os.path.join(ROOT, "profiles", f"{kernel}.traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        sources = rec["source"] if isinstance(rec["source"], list) else [rec["source"]]
        h = hashlib.sha256()
        for src in sources:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        sha = h.hexdigest()
    except (OSError, KeyError, ValueError):
        return None
    if sha != rec.get("source_sha256") or workload != rec.get("bench_workload", "layer"):
        return None
    return int(rec["dram_bytes_per_launch"])


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
            return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---- CPU oracle leg ------------------------------------------------------------------

ORACLE_SLICE = 1 << 21  # weights per oracle container


def oracle_sample(tensors, count: int, slice_elems: int = ORACLE_SLICE):
    """Containers for the CPU oracle: the first `count` full slices of
    slice_elems weights of the workload's tensors (an iterable of (element
    patterns, format), read only as far as needed), in order, each encoded
    as its own container by the oracle's own encoder (equal slices, so that
    every thread gets the same work; the norm vectors, shorter than a slice,
    are left out).  Nothing of the library is loaded for them."""
    import oracle
    work, short = [], []
    for w, fmt in tensors:
        w = w.reshape(-1)
        if w.size < slice_elems and len(short) < max(1, count):
            short.append((w, int(fmt)))
        for s in range(0, w.size - slice_elems + 1, slice_elems):
            if len(work) < count:
                work.append((w[s:s + slice_elems], int(fmt)))
        if len(work) >= count:
            break
    if not work:  # every tensor is shorter than a slice: the tensors themselves
        work = [t for t in short if t[0].size]

    def enc(a):
        w, fmt = a
        return oracle.encode(w, oracle.code_lengths(oracle.histogram(w, fmt)), fmt=fmt)

    with cf.ThreadPoolExecutor(16) as ex:
        return list(ex.map(enc, work))


def part_tensors(parts):
    """(element patterns, format) of each encoded tensor, for oracle_sample."""
    return ((w, d.format) for _, w, _, d in parts)


def time_oracle(containers, threads: int) -> tuple[float, int]:
    """Seconds for the oracle to decode every container on `threads` threads
    (ctypes releases the GIL, so the C decoder runs in parallel)."""
    import oracle
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        results = list(ex.map(oracle.decode, containers))
    dt = time.perf_counter() - t0
    assert all(st == oracle.OK for _, st in results)
    return dt, sum(out.size for out, _ in results)


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


# ---- reference arm (the CPU oracle) ----------------------------------------------------

def run_reference(args):
    rank, world, _ = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0
    if rank != 0:
        return  # rank 0 alone runs the CPU reference
    gens = workload_generators(args.seed, 0, args.workload)
    fmt = FMT_OF_WORKLOAD.get(args.workload, 0)
    threads = os.cpu_count() or 1
    # one step = the oracle restoring a bounded sample: one slice per host
    # thread, from the workload's first tensors (generated only as far as
    # needed; the oracle encodes them itself)
    per_step = oracle_sample(((np.ascontiguousarray(g()), fmt) for g in gens.values()), threads)
    n_total = workload_weights(args.workload)
    threads = max(1, min(threads, len(per_step)))
    for _ in range(args.warmup):
        time_oracle(per_step, threads)
    times, weights = [], 0
    for _ in range(args.steps):
        dt, nw = time_oracle(per_step, threads)
        times.append(dt)
        weights = nw
    sec = sum(times) / len(times)
    value = elem_bytes(fmt) * weights / sec / 1e9
    sample = (f"{len(per_step)} oracle containers ({weights} weights) per step, one per thread, "
              f"from the workload's {n_total} weights")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": workload_text(args.workload), "weights_per_step": weights},
        "weights_per_s": weights / sec,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- our arm ---------------------------------------------------------------------------

def workload_weights(workload: str) -> int:
    """Weights of a workload, from its shapes alone."""
    from weight_streaming_canonical_gb300 import synth
    if workload == "model":
        return synth.model_weight_count()
    if workload in ("layer", "layer-fp16"):
        return synth.layer_weight_count()
    if workload == "layer-e4m3":
        return sum(synth.numel(s) for _, s, k in synth.LAYER_TENSORS if k == "matrix")
    if workload == "matrix4096":
        return 4096 * 4096
    if workload == "adversarial":
        return 1 << 28
    if workload.startswith("normal:"):
        return 1 << int(workload.split(":", 1)[1])
    if workload.startswith("tensor:"):
        name = workload.split(":", 1)[1]
        return synth.numel(dict((n, s) for n, s, _ in synth.LAYER_TENSORS)[name])
    raise SystemExit(f"unknown workload {workload}")


def restore_traffic(kernel: str, workload: str, n_weights: int):
    """DRAM bytes per step of the restore kernel: the committed capture of
    this workload, else, for the whole model (too large to capture, 23
    launches a step), the layer capture's bytes scaled by weights (the
    restore's traffic is proportional to the weights: every tensor has the
    layer's bits per weight).  None when no valid capture exists."""
    t = profiled_traffic(kernel, workload)
    if t is not None or workload != "model":
        return t, "ncu capture of this workload, one launch"
    t = profiled_traffic(kernel, "layer")
    if t is None:
        return None, None
    from weight_streaming_canonical_gb300 import synth
    return int(t * n_weights / synth.layer_weight_count()), \
        "ncu capture of the layer (one launch) scaled to the step by weights"


def measure_restore(afx, parts, dev, args, workload: str, world: int = 1, local: int = 0, clocks: bool = False):
    """Uploads the workload's containers to HBM, checks one graph replay
    of its afx_decode_batch call bit for bit against the original elements
    on the device, then times `args.steps` replays.  Workloads whose bytes
    fit in L2 are timed replay by replay with L2 flushed (a 512 MB write)
    before each, outside the events; larger ones back to back.  With
    `clocks`, the timed replays sit inside about BUSY_PAD_S seconds of the
    same work on each side while nvidia-smi samples the clocks.  Returns
    (result, state) with state holding the device buffers for later legs."""
    import torch
    n_total = sum(d.n for _, _, _, d in parts)
    comp_total = sum(d.container_bytes for _, _, _, d in parts)
    alg_total = sum(algorithmic_bytes(d) for _, _, _, d in parts)
    offs, o = [], 0
    for _, _, c, _ in parts:
        offs.append(o)
        o += c.size
    host_blob = torch.empty(o, dtype=torch.uint8).pin_memory()
    hb = host_blob.numpy()
    for (_, _, c, _), off in zip(parts, offs):
        hb[off:off + c.size] = c
    dev_blob = host_blob.to(dev)
    out_offs, oo = [], 0
    for _, _, _, d in parts:
        out_offs.append(oo)
        oo += d.n
    fmt = fmt_of(parts)
    out = torch.empty(oo, dtype=torch_elem_dtype(fmt), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    views = [(d, dev_blob[off:off + d.container_bytes], out[oo_:oo_ + d.n])
             for (_, _, _, d), off, oo_ in zip(parts, offs, out_offs)]
    descs = [d for d, _, _ in views]
    # kernel launches one afx_decode_batch call makes: up to 16 coded tensors
    # per restore launch, one fill launch per single-exponent tensor
    coded = sum(1 for d in descs if d.nsym >= 2 and d.n)
    launches_per_step = (coded + 15) // 16 + sum(1 for d in descs if d.nsym == 1 and d.n)
    cviews = [c for _, c, _ in views]
    oviews = [o for _, _, o in views]
    # chunks a lane of the step's restore launches (the kernel that runs)
    lanes = max(afx.afx_decode_chunks_a_lane(descs, cviews) + [0])

    def step():
        afx.afx_decode_batch(descs, cviews, oviews, status_dev=status)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()
    # correctness of what is timed: the restored elements equal the original bits
    with torch.cuda.stream(stream):
        out.zero_()
        graph.replay()
    torch.cuda.synchronize()
    for (name, w, _, _), oo_ in zip(parts, out_offs):  # compared on the device, one tensor at a time
        ref = torch.from_numpy(w.view(np.uint8 if fmt == 2 else np.int16)).to(dev)
        if not torch.equal(out[oo_:oo_ + w.size], ref):
            raise SystemExit(f"restore of {name} is not bit-exact")
        del ref
    if status.item() != 0:
        raise SystemExit(f"device status {status.item()}")

    small = comp_total + elem_bytes(fmt) * n_total < 2 * L2_BYTES
    flush = torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=dev) if small else None

    def one_step():
        if small:
            flush.fill_(1)
        graph.replay()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    pad, sampler = 0, None
    if clocks:
        est0, est1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            est0.record(stream)
            for _ in range(3):
                one_step()
            est1.record(stream)
        torch.cuda.synchronize()
        pad = busy_pad_steps(est0.elapsed_time(est1) / 3)
        barrier(world)
        sampler = ClockSampler(local)
        time.sleep(0.3)
    torch.cuda.synchronize()
    busy_t0 = time.time()
    with torch.cuda.stream(stream):
        for _ in range(pad):
            one_step()
    if small:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                flush.fill_(1)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            for _ in range(pad):
                one_step()
        torch.cuda.synchronize()
        ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / args.steps
    else:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(args.steps):
                graph.replay()
            end.record(stream)
            for _ in range(pad):
                one_step()
        torch.cuda.synchronize()
        ms = start.elapsed_time(end) / args.steps
    busy_t1 = time.time()
    clk = sampler.stop((busy_t0, busy_t1)) if sampler is not None else None
    if clk is not None:
        clk["busy_pad_steps_each_side"] = pad
    barrier(world)
    ms = max_over_ranks(ms, world)

    # The graph holds the step's restore launches and nothing else, so its
    # replay time bounds their summed duration from above: the kernel's
    # time per step is taken in that same window.
    peak, peak_kind = measured_hbm_peak()
    achieved = alg_total / (ms * 1e-3) / 1e9
    kernel_name = {1: "restore_store_fp16_kernel", 2: "restore_store_e4m3_kernel"}.get(fmt, "restore_store_kernel")
    if lanes == 2:  # two chunks a lane
        kernel_name = kernel_name.replace("_kernel", "_pair_kernel")
    traffic, traffic_src = restore_traffic(kernel_name, workload, n_total)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "traffic_scope": "per step" + (f" ({traffic_src})" if traffic_src else ""),
                "kernel": kernel_name, "chunks_a_lane": lanes, "peak_kind": peak_kind,
                "launches_per_step": launches_per_step, "algorithmic_bytes_per_step": alg_total,
                "kernel_ms_per_step": ms,
                "kernel_time": "graph replays holding only the restore launches (the launches' summed duration "
                               "is at most this)"}
    res = {"ms": ms, "n": n_total, "comp": comp_total, "alg": alg_total, "fmt": fmt, "small": small,
           "roofline": roofline, "clocks": clk, "launches_per_step": launches_per_step, "bit_exact": True,
           "tensors": len(views)}
    state = {"dev_blob": dev_blob, "offs": offs, "views": views, "host_blob": host_blob, "out": out}
    return res, state


def config_summary(workload: str, res: dict) -> dict:
    """One workload's restore result for the per_config block."""
    sec = res["ms"] * 1e-3
    return {"workload": workload_text(workload), "weights": res["n"], "ms_per_step": res["ms"],
            "weights_per_s": res["n"] / sec, "decoded_gbs": elem_bytes(res["fmt"]) * res["n"] / sec / 1e9,
            "hbm_gbs": res["alg"] / sec / 1e9, "hbm_frac": res["roofline"]["frac"],
            "peak_kind": res["roofline"]["peak_kind"], "bit_exact": res["bit_exact"],
            "launches_per_step": res["launches_per_step"], "bits_per_weight": 8 * res["comp"] / res["n"],
            "l2": "flushed before each timed replay" if res["small"] else "inputs larger than L2"}


PER_CONFIG = (("1", "matrix4096"), ("2", "layer"), ("3", "model"), ("4", "adversarial"))


def run_ours(args):
    import torch

    from weight_streaming_canonical_gb300 import afx

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    parts = build_layer(args.seed, rank, args.workload)
    res, state = measure_restore(afx, parts, dev, args, args.workload, world, local, clocks=True)
    ms, n_total, comp_total, alg_total, fmt = res["ms"], res["n"], res["comp"], res["alg"], res["fmt"]
    peak = res["roofline"]["peak"]
    sec = ms * 1e-3
    value, weights_per_s = job_throughput(n_total, world, ms, elem_bytes(fmt))
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32",
        "data": data_text(args.workload),
        "config": {"workload": workload_text(args.workload), "weights": n_total, "compressed_bytes": comp_total,
                   "bits_per_weight": 8 * comp_total / n_total,
                   "coded_exponent_bits_per_weight": sum(d.total_bits for *_, d in parts) / n_total,
                   "exponent_entropy_bits_per_weight": exponent_entropy_bits(parts),
                   "l2": ("L2 flushed before each timed launch (a 512 MB write outside the events): "
                          if res["small"] else "inputs larger than L2: ")
                         + "%.0f MB compressed read and %.0f MB written per step"
                         % (comp_total / 1e6, elem_bytes(fmt) * n_total / 1e6),
                   "launch": f"one afx_decode_batch call of {res['tensors']} tensors "
                             f"({res['launches_per_step']} kernel launches) per step, replayed from a CUDA graph",
                   "parallelism": f"replicas x{world}"},
        "weights_per_s": weights_per_s,
        "hbm_gbs": alg_total * world / sec / 1e9,
        "hbm_frac": alg_total / sec / 1e9 / peak,
        "hbm_frac_of_nominal_7900_gbs": alg_total / sec / 1e9 / 7900.0,
        "roofline": res["roofline"],
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": res["clocks"],
    }

    legs = set(args.legs.split(",")) if args.legs != "all" else {
        "e2e", "zero_copy", "cpu_baseline", "gemv", "stream", "prefill", "formats", "encode", "configs", "wide_trees"}
    if not args.no_extras and "e2e" in legs:
        # every rank runs the end-to-end leg on its own GPU and host link; the
        # job's figure is all ranks' bytes over the slowest rank's time
        e2e = run_e2e(afx, parts, state["views"], dev, args, host_blob=state["host_blob"], offs=state["offs"])
        e2e_ms = max_over_ranks(e2e["ms_per_step"], world)
        e2e["value"] = e2e["value"] * world * e2e["ms_per_step"] / e2e_ms
        e2e["ms_per_step"] = e2e_ms
        e2e["h2d_bytes_per_step"] *= world
        e2e["d2h_bytes_per_step"] *= world
        if world > 1:
            e2e["ranks"] = world
        line["e2e"] = e2e
    extras = not args.no_extras and rank == 0 and world == 1  # the other legs and the CPU oracle at N = 1 only
    if extras and "cpu_baseline" in legs:
        line["cpu_baseline"] = run_cpu_baseline(parts)
    layer_parts, layer_state, layer_value = None, None, None
    if args.workload == "layer":
        layer_parts, layer_state, layer_value = parts, state, value
    else:
        del state
    del parts
    if extras and "configs" in legs:
        # every other config of the method's workloads, each bit-exact checked
        # before it is timed; the headline's own entry repeats its numbers
        per = {}
        for key, wl in PER_CONFIG:
            if wl == args.workload:
                per[key] = config_summary(wl, res)
                continue
            p = build_layer(args.seed, 0, wl)
            r, st = measure_restore(afx, p, dev, args, wl)
            per[key] = config_summary(wl, r)
            if wl == "layer":
                layer_parts, layer_state, layer_value = p, st, elem_bytes(r["fmt"]) * r["n"] / (r["ms"] * 1e-3) / 1e9
                per[key]["note"] = "the layer's extra legs below use these containers"
            else:
                del p, st
            torch.cuda.empty_cache()
        line["per_config"] = per
    if extras and layer_parts is None and legs & {"zero_copy", "encode", "gemv", "stream", "prefill"}:
        layer_parts = build_layer(args.seed, 0, "layer")
        r, layer_state = measure_restore(afx, layer_parts, dev, args, "layer")
        layer_value = elem_bytes(r["fmt"]) * r["n"] / (r["ms"] * 1e-3) / 1e9
    if extras:
        parts = layer_parts
        dev_blob, offs = (layer_state["dev_blob"], layer_state["offs"]) if layer_state else (None, None)
        lw = sum(d.n for *_, d in parts) if parts else 0
        if "zero_copy" in legs:
            line["zero_copy"] = run_zero_copy(afx, parts, dev, args)
        if "encode" in legs:
            line["host_encode"] = run_host_encode(afx, parts)
        if "gemv" in legs:
            line["fused_gemv"] = run_gemv_bench(afx, parts, dev_blob, offs, dev, args,
                                                layer_value * 1e9 / 2 if layer_value else None)
        if "stream" in legs:
            line["streamed_40_layers"] = run_stream_bench(afx, parts, dev, args)
            # "Why Weight Offloading Slows Inference", Eq. (2): compression pays
            # when (S - S_disk) / b > t_unpack; here b is the measured link
            S, S_disk = 2 * lw, sum(d.container_bytes for *_, d in parts)
            b = line["streamed_40_layers"]["batch1"]["h2d_gbs"] * 1e9
            t_unpack_ms = 2 * lw / (layer_value * 1e9) * 1e3
            line["eq2_break_even"] = {"S_bytes": S, "S_disk_bytes": S_disk, "b_link_gbs": b / 1e9,
                                      "read_time_saved_ms": (S - S_disk) / b * 1e3, "t_unpack_ms": t_unpack_ms,
                                      "pays": (S - S_disk) / b > t_unpack_ms * 1e-3,
                                      "scope": "one Qwen3-14B-shaped layer"}
            line["residency_plan"] = run_residency_plan(afx, parts, b / 1e9, layer_value)
        if "prefill" in legs:
            line["prefill"] = run_prefill_bench(afx, parts, dev_blob, offs, dev, args)
        if "gemv" in legs and "prefill" in legs:
            line["fused_gemv"]["vs_restore_then_gemm"] = fused_vs_unfused(line["fused_gemv"], line["prefill"])
        if "formats" in legs:
            line["formats"] = run_formats_bench(afx, dev, args)
        if "wide_trees" in legs:
            line["wide_trees"] = run_wide_trees_bench(afx, dev, args, layer_value * 1e9 / 2 if layer_value else None)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_host_encode(afx, parts, reps: int = 2):
    """The host side of the method, timed: the step's tensors encoded through
    the C ABI (exponent histogram, length-limited canonical code, packing of
    the stream and both indices), one tensor after another, each encode
    spread over the host's threads.  Best of `reps`; the containers must
    equal the ones the step restores."""
    fmt = fmt_of(parts)
    best = None
    for _ in range(reps):
        t0 = time.perf_counter()
        out = [afx.encode(w, fmt=fmt)[0] for _, w, _, _ in parts]
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    same = all(np.array_equal(o, c) for o, (_, _, c, _) in zip(out, parts))
    n = sum(w.size for _, w, _, _ in parts)
    return {"ms": best * 1e3, "weights_per_s": n / best, "input_gbs": elem_bytes(fmt) * n / best / 1e9,
            "host_threads": os.cpu_count(), "containers_identical": bool(same),
            "path": "afx.encode per tensor (afx_build_code_fmt, afx_encode_bound, afx_encode), host only"}


def run_e2e(afx, parts, views, dev, args, host_blob=None, offs=None):
    """Pinned host containers -> device -> BF16 back to pinned host, through
    afx_stream_run with one tensor per streamed layer: the copy of tensor
    i+1 overlaps the restore of tensor i, and the copy back of tensor i
    (on its own stream) overlaps both.  host_blob/offs: the containers
    already in pinned host memory, back to back (used as they are)."""
    import torch
    fmt = fmt_of(parts)
    host_out = torch.empty(sum(d.n for _, _, _, d in parts), dtype=torch_elem_dtype(fmt)).pin_memory()
    blobs, ops_all, outs = [], [], []
    o = 0
    piece = args.e2e_piece_weights
    if piece > 0:  # the same weights as consecutive slices, one container each
        sliced = []
        for (name, w, _, _) in parts:
            flat = w.reshape(-1)
            for i in range(0, max(flat.size, 1), piece):
                c, d = afx.encode(flat[i:i + piece], fmt=fmt)
                sliced.append((name, flat[i:i + piece], c, d))
        stream_parts = sliced
    else:
        stream_parts = parts
    for i, (_, w, c, d) in enumerate(stream_parts):
        if piece <= 0 and host_blob is not None:
            blob = host_blob[offs[i]:offs[i] + c.size]
        else:
            blob = torch.empty(c.size, dtype=torch.uint8).pin_memory()
            blob.numpy()[:] = c
        out = torch.empty(d.n, dtype=torch_elem_dtype(fmt), device=dev)
        op = afx.afx_op()
        op.desc = d
        op.offset = 0
        op.kind = afx.AFX_OP_DECODE
        op.out_dev = out.data_ptr()
        op.out_host = host_out[o:o + d.n].data_ptr()
        o += d.n
        blobs.append(blob)
        ops_all.append([op])
        outs.append(out)
    buf_bytes = max(b.numel() for b in blobs)
    bufs = [torch.empty(buf_bytes, dtype=torch.uint8, device=dev) for _ in range(3)]
    compute, copy, d2h = (torch.cuda.Stream(device=dev) for _ in range(3))
    layers = list(zip(blobs, ops_all))

    def step():
        compute.wait_stream(d2h)  # the previous step's copies back have read the outputs
        afx.afx_stream_run(layers, bufs, buf_bytes, compute, copy, d2h_stream=d2h)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    steps = max(3, args.steps // 2)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(compute)
    for _ in range(steps):
        step()
    compute.wait_stream(d2h)
    end.record(compute)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    n = sum(d.n for _, _, _, d in stream_parts)
    eb = elem_bytes(fmt)
    ws_ = [w.reshape(-1) for _, w, _, _ in stream_parts]
    ok = all(np.array_equal(host_out.numpy().view(np_elem_dtype(fmt))[s:s + w.size], w)
             for s, w in zip(np.cumsum([0] + [w.size for w in ws_])[:-1], ws_))
    return {"value": eb * n / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(sum(b.numel() for b in blobs)), "d2h_bytes_per_step": eb * n,
            "bit_exact": bool(ok), "containers": len(stream_parts),
            "path": ("afx_stream_run, one container per streamed stage"
                     + (f" (each tensor stored as slices of at most {piece} weights)" if piece > 0 else
                        " (one per tensor)")
                     + ": pinned host containers in, BF16 back to pinned host on a third stream")}


def run_zero_copy(afx, parts, dev, args):
    """The layer's containers stay in pinned host memory and one
    afx_decode_batch call reads them over the host link (no staging copy):
    into device memory, and back into pinned host memory (host to host in
    one launch).  Compared with the copy pipeline in e2e."""
    import torch
    n = sum(d.n for _, _, _, d in parts)
    fmt = fmt_of(parts)
    eb = elem_bytes(fmt)
    host_c = []
    for (_, _, c, _) in parts:
        t = torch.empty(c.size, dtype=torch.uint8).pin_memory()
        t.numpy()[:] = c
        host_c.append(t)
    descs = [d for *_, d in parts]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {}
    for where in ("device", "host"):
        if where == "device":
            outs = [torch.empty(d.n, dtype=torch_elem_dtype(fmt), device=dev) for d in descs]
        else:
            outs = [torch.empty(d.n, dtype=torch_elem_dtype(fmt)).pin_memory() for d in descs]
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                afx.afx_decode_batch(descs, host_c, outs, stream=stream, status_dev=status)
            torch.cuda.synchronize()
            steps = max(3, args.steps // 2)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                afx.afx_decode_batch(descs, host_c, outs, stream=stream, status_dev=status)
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        ok = status.item() == 0 and all(np.array_equal(o.cpu().numpy().view(np_elem_dtype(fmt)), w)
                                        for o, (_, w, _, _) in zip(outs, parts))
        res["to_" + where] = {"value": eb * n / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
                              "link_read_bytes": int(sum(c.numel() for c in host_c)),
                              "link_write_bytes": eb * n if where == "host" else 0, "bit_exact": bool(ok)}
    res["path"] = ("afx_decode_batch of the layer with its containers in pinned host memory, read by "
                   "restore_store_host_kernel over the host link; to_host also writes the BF16 weights to "
                   "pinned host memory")
    return res


def run_prefill_bench(afx, parts, dev_blob, offs, dev, args):
    """The layer's seven matrices times N token vectors (prefill), containers
    resident in HBM: restore then tensor-core product per matrix on one
    stream, the same with restores overlapped with products on two streams
    (afx_prefill_batch), and the restores alone."""
    import torch
    from weight_streaming_canonical_gb300 import synth
    shapes = {name: shape for name, shape, _ in synth.LAYER_TENSORS}
    mats = [(name, d, int(off)) for (name, _, _, d), off in zip(parts, offs) if len(shapes.get(name, ())) == 2]
    n_w = sum(d.n for _, d, _ in mats)
    biggest = max(d.n for _, d, _ in mats)
    scratch = [torch.empty(biggest, dtype=torch.int16, device=dev) for _ in range(2)]
    ws = torch.empty(afx.AFX_PREFILL_GEMM_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
    conts = [dev_blob[off:off + d.container_bytes] for _, d, off in mats]
    descs = [d for _, d, _ in mats]
    mshapes = [shapes[name] for name, _, _ in mats]
    peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"] if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0
    rs, gs = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    out = {"matrices": len(mats), "weights": n_w, "bf16_peak_tflops": peak, "runs": []}

    def timed(fn, stream, reps=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    padded = [(d.n * 2 + 255) // 256 * 128 for d in descs]
    whole = torch.empty(sum(padded), dtype=torch.int16, device=dev)
    whole_views = [whole[o:o + d.n] for o, d in zip(np.cumsum([0] + padded[:-1]), descs)]
    with torch.cuda.stream(gs):
        def restores():
            for (_, d, _), c in zip(mats, conts):
                afx.afx_decode(d, c, scratch[0][:d.n], stream=gs)
        restore_ms = timed(restores, gs)
        restore_one_launch_ms = timed(lambda: afx.afx_decode_batch(descs, conts, whole_views, stream=gs), gs)
    out["restore_ms_per_matrix_launches"] = restore_ms
    out["restore_ms_one_launch"] = restore_one_launch_ms
    # the same matrices in tile order for the fused product (encoded on the host)
    shape_of = {name: shapes[name] for name, _, _ in mats}
    w_of = {name: w for name, w, _, _ in parts}

    def tiled(name):
        r, cl = shape_of[name]
        return afx.encode(afx.afx_tile_order(w_of[name], r, cl))

    with cf.ThreadPoolExecutor(len(mats)) as ex:
        tiled_parts = list(ex.map(tiled, [name for name, _, _ in mats]))
    tdescs = [d for _, d in tiled_parts]
    tconts = [torch.from_numpy(c).to(dev) for c, _ in tiled_parts]
    fused_ws = torch.empty(afx.afx_prefill_fused_workspace(), dtype=torch.uint8, device=dev)
    out["fused_workspace_bytes"] = fused_ws.numel()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for n_tok in (1, 4, 128, 512, 2048):
        reps = 20 if n_tok <= 4 else 5
        xs = [torch.from_numpy(synth.activations(n_tok, cl, seed=21).view(np.int16)).to(dev) for _, cl in mshapes]
        ys = [torch.empty((n_tok, r), dtype=torch.float32, device=dev) for r, _ in mshapes]
        yf = [torch.empty((n_tok, r), dtype=torch.float32, device=dev) for r, _ in mshapes]

        def sequential():
            for i, (d, c) in enumerate(zip(descs, conts)):
                r, cl = mshapes[i]
                afx.afx_prefill(d, c, r, cl, xs[i], ys[i], scratch[0], ws, stream=gs)

        def overlapped():
            afx.afx_prefill_batch(descs, conts, mshapes, xs, ys, scratch, ws, restore_stream=rs, gemm_stream=gs)

        def one_launch():
            afx.afx_prefill_batch(descs, conts, mshapes, xs, ys, [whole, None], ws, gemm_stream=gs)

        def fused():
            afx.afx_prefill_fused_batch(tdescs, tconts, mshapes, xs, yf, fused_ws, stream=gs, status_dev=status)

        seq_ms = timed(sequential, gs, reps)
        ovl_ms = timed(overlapped, gs, reps)
        one_ms = timed(one_launch, gs, reps)
        fused_ms = timed(fused, gs, reps)
        # the fused products against the unfused ones (cuBLAS over the
        # restored weights), per output within 2 x 2e-3 * sum|w x| (each side
        # is within 2e-3 of the exact sum); the bound from a float32 product
        # of the absolute values
        with torch.cuda.stream(gs):
            one_launch()
            fused()
        torch.cuda.synchronize()
        agree, worst = status.item() == 0, 0.0
        for i, (r, cl) in enumerate(mshapes):
            wv = whole_views[i]
            wabs = (wv.view(torch.bfloat16).float().abs()).view(r, cl)
            bound = xs[i].view(torch.bfloat16).float().abs() @ wabs.t()
            err = (yf[i] - ys[i]).abs()
            worst = max(worst, float((err / bound.clamp_min(1e-30)).max()))
            agree = agree and bool((err <= 4e-3 * bound + 1e-30).all())
            del wabs, bound, err
        gemm_ms = max(seq_ms - restore_ms, 1e-9)
        best = min(seq_ms, ovl_ms, one_ms)
        flop = 2.0 * n_w * n_tok
        out["runs"].append({"tokens": n_tok, "sequential_ms": seq_ms, "overlapped_ms": ovl_ms,
                            "one_restore_launch_ms": one_ms, "gemm_ms_from_difference": gemm_ms,
                            "tokens_per_s": n_tok / (best * 1e-3), "tflops": flop / (best * 1e-3) / 1e12,
                            "gemm_tflops": flop / (gemm_ms * 1e-3) / 1e12,
                            "gemm_frac_of_bf16_peak": flop / (gemm_ms * 1e-3) / 1e12 / peak,
                            "best_over_sum_of_parts": best / (restore_one_launch_ms + gemm_ms),
                            "fused_ms": fused_ms, "fused_tokens_per_s": n_tok / (fused_ms * 1e-3),
                            "fused_tflops": flop / (fused_ms * 1e-3) / 1e12,
                            "fused_weights_per_s": n_w * ((n_tok + 511) // 512) / (fused_ms * 1e-3),
                            "unfused_best_over_fused": best / fused_ms,
                            "fused_agrees_with_unfused": agree, "fused_worst_err_over_sum_abs": worst})
    out["path"] = ("afx_prefill / afx_prefill_batch: the restore (restore_store_pair_kernel for a launch of the "
                   "seven matrices, two chunks a lane) into scratch, cuBLAS BF16 GEMM with "
                   "float32 accumulation; sequential: restore then product per matrix on one stream; overlapped: "
                   "restore of matrix i+1 on a second stream; one restore launch: all seven restored by one "
                   "afx_decode_batch launch, then the products; tokens_per_s and tflops from the fastest of "
                   "those; fused: afx_prefill_fused_batch over the tile-ordered containers (prefill_fused_kernel: "
                   "restored 128x64 tiles through a 256 KB ring per SM that stays in L2, TMA into shared memory, "
                   "tcgen05 products, no restored matrix written out; the weights are restored once per 512 "
                   "tokens, counted in fused_weights_per_s)")
    return out


def fused_vs_unfused(fused: dict, prefill: dict) -> dict:
    """The fused product against the unfused path at the same batch: all
    seven matrices restored to BF16 in HBM scratch, then cuBLAS products
    (afx_prefill_batch, fastest of its three forms).  ratio > 1: the fused
    product is faster."""
    runs = {r["tokens"]: r for r in prefill.get("runs", [])}
    out = {}
    for B in (1, 4):
        f, r = fused.get(f"batch{B}"), runs.get(B)
        if not f or not r:
            continue
        form, unfused = min((("sequential", r["sequential_ms"]), ("overlapped", r["overlapped_ms"]),
                             ("one_restore_launch", r["one_restore_launch_ms"])), key=lambda kv: kv[1])
        out[f"batch{B}"] = {"fused_ms": f["ms"], "restore_then_gemm_ms": unfused, "unfused_form": form,
                            "unfused_over_fused": unfused / f["ms"]}
    return out


def run_formats_bench(afx, dev, args):
    """The other element formats on the same layer shapes, containers resident
    in HBM, one afx_decode_batch launch per step: FP16 (all nine tensors, the
    BF16 distributions rounded to FP16) and E4M3 (the seven matrices with a
    per-tensor scale).  Bit-exact check first, then the median of per-launch
    CUDA-event times."""
    import torch
    from weight_streaming_canonical_gb300 import synth
    out = {}
    for fmt, label in ((afx.AFX_FMT_FP16, "fp16"), (afx.AFX_FMT_E4M3, "e4m3")):
        if fmt == afx.AFX_FMT_FP16:
            gens = [(nm, (lambda nm=nm: synth.layer_tensor_fp16(nm, seed=args.seed))) for nm, _, _ in synth.LAYER_TENSORS]
        else:
            gens = [(nm, (lambda nm=nm: synth.layer_matrix_e4m3(nm, seed=args.seed)))
                    for nm, _, kind in synth.LAYER_TENSORS if kind == "matrix"]

        def one(item, fmt=fmt):
            nm, gen = item
            w = np.ascontiguousarray(gen()).reshape(-1)
            c, d = afx.encode(w, fmt=fmt)
            return nm, w, c, d

        with cf.ThreadPoolExecutor(min(len(gens), 16)) as ex:
            parts = list(ex.map(one, gens))
        elem = afx.element_bytes(fmt)
        descs = [d for *_, d in parts]
        conts = [torch.from_numpy(c).to(dev) for _, _, c, _ in parts]
        outs = [torch.empty(w.size, dtype=torch.uint8 if elem == 1 else torch.int16, device=dev) for _, w, _, _ in parts]
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            afx.afx_decode_batch(descs, conts, outs, stream=stream, status_dev=status)
        torch.cuda.synchronize()
        exact = status.item() == 0 and all(
            torch.equal(o, torch.from_numpy(w.view(np.uint8 if elem == 1 else np.int16)).to(dev))
            for (_, w, _, _), o in zip(parts, outs))
        reps = max(10, args.steps)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(stream):
            for _ in range(3):
                afx.afx_decode_batch(descs, conts, outs, stream=stream, status_dev=status)
            for e0, e1 in ev:
                e0.record(stream)
                afx.afx_decode_batch(descs, conts, outs, stream=stream, status_dev=status)
                e1.record(stream)
        torch.cuda.synchronize()
        ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
        n = sum(d.n for d in descs)
        alg = sum(algorithmic_bytes(d) for d in descs)
        comp = sum(d.container_bytes for d in descs)
        peak, peak_kind = measured_hbm_peak()
        sym_bits = 0.0
        for _, w, _, d in parts:
            sym = (w >> 3) & 0xF if elem == 1 else (w >> 10) & 0x1F if fmt == afx.AFX_FMT_FP16 else (w >> 7) & 0xFF
            cnt = np.bincount(sym.astype(np.intp), minlength=256).astype(np.float64)
            p = cnt[cnt > 0] / w.size
            sym_bits += float(-(p * np.log2(p)).sum()) * w.size
        out[label] = {
            "tensors": len(parts), "elements": n, "bit_exact": bool(exact), "ms": ms,
            "decoded_gbs": elem * n / (ms * 1e-3) / 1e9, "elements_per_s": n / (ms * 1e-3),
            "hbm_gbs": alg / (ms * 1e-3) / 1e9, "hbm_frac": alg / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
            "bits_per_element": 8 * comp / n, "raw_bits_per_element": 8 * elem,
            "coded_symbol_bits_per_element": sum(d.total_bits for d in descs) / n,
            "symbol_entropy_bits_per_element": sym_bits / n,
            "algorithmic_bytes_per_step": alg,
        }
    out["path"] = ("afx_decode_batch of the whole set per step: restore_store_fp16_kernel (raw bytes plus the hi "
                   "section) and restore_store_e4m3_kernel (raw nibbles, byte outputs)")
    return out


WIDE_TREES = ((51, 0.85), (52, 0.85), (57, 0.85), (80, 0.9), (100, 0.92), (120, 0.94))
def run_wide_trees_bench(afx, dev, args, layer_weights_per_s=None):
    """Restore rate against the size of the code tree: one 2^27-weight tensor
    per exponent mix (geometric exponent frequencies, synth.exponent_mix),
    and one N(0, 0.02) tensor with rare exponents across the whole range;
    each restored by one launch, bit-exact checked, then timed.  The decoder
    each one gets comes from afx_decode_table_kind: the whole byte-step
    state table while its rows fit (50 internal nodes beside 32 warps
    staging 16-byte chunks), beyond that rows for the shallowest nodes plus
    escapes."""
    from weight_streaming_canonical_gb300 import synth
    kinds = {afx.AFX_TABLE_FILL: "fill", afx.AFX_TABLE_LUT12: "12-bit multi-code table",
             afx.AFX_TABLE_STATES: "byte-step state table, every node",
             afx.AFX_TABLE_PARTIAL: "byte-step state table, shallowest nodes + escapes"}
    out = {"weights": 1 << 27, "runs": []}
    cases = [(f"mix{n_exp}", n_exp, ratio) for n_exp, ratio in WIDE_TREES] + [("tail", None, None)]
    for label, n_exp, ratio in cases:
        if n_exp is None:
            w = synth.long_tail(1 << 27, seed=3)
        else:
            w = synth.exponent_mix(1 << 27, n_exp, ratio=ratio, seed=n_exp)
        c, d = afx.encode(w)
        kind, rows = afx.afx_decode_table_kind(d)
        r, st = measure_restore(afx, [(label, w, c, d)], dev, args, f"{label}")
        del st
        wps = r["n"] / (r["ms"] * 1e-3)
        out["runs"].append({"case": label, "exponents": d.nsym, "internal_nodes": d.nsym - 1,
                            "ratio": ratio, "ms": r["ms"], "weights_per_s": wps,
                            "hbm_frac": r["roofline"]["frac"], "bit_exact": r["bit_exact"],
                            "coded_bits_per_weight": d.total_bits / d.n, "chunk_bytes": d.chunk_bytes,
                            "decoder": kinds.get(kind, str(kind)), "state_rows": rows,
                            "frac_of_layer_rate": wps / layer_weights_per_s if layer_weights_per_s else None})
        del w, c
    out["path"] = ("afx_decode_batch of one tensor per step (restore_store_kernel, restore_store_pair_kernel where "
                   "two chunks a lane fit beside the tables, or restore_store_partial_kernel for a partial state "
                   "table)")
    return out


def run_residency_plan(afx, parts, link_gbs, restore_gbs):
    """afx_plan_residency for the whole Qwen3-14B-shaped model (40 layers
    with this layer's container sizes, embedding and head at the matrices'
    bits per weight) with the link and restore rates measured in this run,
    at device budgets from the pages' 8 GB laptop GPU upwards."""
    from weight_streaming_canonical_gb300 import synth
    tensors = [(2 * d.n, d.container_bytes) for _ in range(synth.LAYERS) for _, _, _, d in parts]
    mats = [d for name, _, _, d in parts if name == "gate_proj"]
    bpw = mats[0].container_bytes / mats[0].n if mats else 1.37
    for shape in (synth.EMBED_SHAPE, synth.HEAD_SHAPE):
        n = synth.numel(shape)
        tensors.append((2 * n, int(n * bpw)))
    names = {afx.AFX_RESIDENT_DECODED: "resident_decoded", afx.AFX_RESIDENT_COMPRESSED: "resident_compressed",
             afx.AFX_STREAM_COMPRESSED: "stream_compressed", afx.AFX_STREAM_RAW: "stream_raw"}
    out = {"link_gbs": link_gbs, "restore_gbs": restore_gbs, "tensors": len(tensors),
           "model_bf16_bytes": sum(S for S, _ in tensors), "model_compressed_bytes": sum(C for _, C in tensors),
           "plans": []}
    for gb in (8, 16, 24, 32):
        place, ms, resident = afx.afx_plan_residency(tensors, gb * 10**9, link_gbs, restore_gbs, overlapped=True)
        counts = {v: place.count(k) for k, v in names.items()}
        out["plans"].append({"budget_gb": gb, "step_ms": ms, "resident_bytes": resident, **counts})
    return out


def _layer_ops(afx, parts, B, dev, keep):
    """Ops for one streamed layer (its containers back to back in one blob):
    the two norms restored, the seven matrices through the fused GEMV with B
    activation rows."""
    import torch
    from weight_streaming_canonical_gb300 import synth
    shapes = {name: shape for name, shape, _ in synth.LAYER_TENSORS}
    kinds = {name: kind for name, _, kind in synth.LAYER_TENSORS}
    offs = np.cumsum([0] + [c.size for _, _, c, _ in parts])[:-1]
    ops = []
    for (name, w, c, d), off in zip(parts, offs):
        op = afx.afx_op()
        op.desc = d
        op.offset = int(off)
        if kinds.get(name) == "norm":
            out = torch.empty(d.n, dtype=torch.int16, device=dev)
            op.kind = afx.AFX_OP_DECODE
            op.out_dev = out.data_ptr()
            keep.append(out)
        else:
            rows, cols = shapes[name]
            x = torch.from_numpy(synth.activations(B, cols, seed=11).view(np.int16)).to(dev)
            y = torch.empty((B, rows), dtype=torch.float32, device=dev)
            ws = torch.empty(afx.afx_decode_gemv_workspace(d, B) // 4 + 4, dtype=torch.float32, device=dev)
            op.kind = afx.AFX_OP_GEMV
            op.rows, op.cols, op.batch = rows, cols, B
            op.x_dev, op.out_dev, op.workspace_dev = x.data_ptr(), y.data_ptr(), ws.data_ptr()
            op.workspace_bytes = ws.numel() * 4
            keep.extend([x, y, ws])
        ops.append(op)
    return ops


def run_gemv_bench(afx, parts, dev_blob, offs, dev, args, restore_weights_per_s=None):
    """Fused restore + GEMV over the layer's seven matrices in one launch,
    batch 1 and 4, containers resident in HBM."""
    import torch
    from weight_streaming_canonical_gb300 import synth
    shapes = {name: shape for name, shape, _ in synth.LAYER_TENSORS}
    res = {}
    mats = [(name, d, off) for (name, _, _, d), off in zip(parts, offs) if name in shapes and len(shapes[name]) == 2]
    n = sum(d.n for _, d, _ in mats)
    comp = sum((d.total_bits + 7) // 8 + d.n + 2 * d.n_chunks + 8 * (d.n_blocks + 1) for _, d, _ in mats)
    for B in (1, 4):
        xs, ys, wss = [], [], []
        for name, d, off in mats:
            rows, cols = shapes[name]
            xs.append(torch.from_numpy(synth.activations(B, cols, seed=5).view(np.int16)).to(dev))
            ys.append(torch.empty((B, rows), dtype=torch.float32, device=dev))
            wss.append(torch.empty(afx.afx_decode_gemv_workspace(d, B) // 4 + 4, dtype=torch.float32, device=dev))
        descs = [d for _, d, _ in mats]
        conts = [dev_blob[off:off + d.container_bytes] for _, d, off in mats]
        shp = [shapes[name] for name, _, _ in mats]
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                afx.afx_decode_gemv_batch(descs, conts, shp, xs, ys, wss)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                afx.afx_decode_gemv_batch(descs, conts, shp, xs, ys, wss)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        # bytes the product must move: the containers' coded bits, sign|mantissa
        # bytes and indices, x read once, y written once
        io = comp + sum(2 * B * c + 4 * B * r for r, c in shp)
        peak, peak_kind = measured_hbm_peak()
        res[f"batch{B}"] = {"ms": ms, "weights_per_s": n / (ms * 1e-3), "compressed_read_gbs": comp / (ms * 1e-3) / 1e9,
                            "hbm_gbs": io / (ms * 1e-3) / 1e9, "hbm_frac": io / (ms * 1e-3) / 1e9 / peak,
                            "peak_kind": peak_kind,
                            "frac_of_restore_rate": (n / (ms * 1e-3)) / restore_weights_per_s
                            if restore_weights_per_s else None,
                            "launches": "one restore kernel (restore_gemv_pair_kernel<1> at batch 1, two chunks a lane; "
                                         "restore_gemv_kernel<4> at batch 4) and one row fix-up per product batch"}
    res["weights"] = n
    res["bound"] = ("the decode's instruction rate (the same byte-step decoder as the restore), not HBM: "
                    "frac_of_restore_rate compares the product's weights/s with the restore's")
    return res


def run_stream_bench(afx, parts, dev, args, layers=40):
    """40 streamed layer steps: compressed layers in pinned host memory, the
    copy of layer l+1 overlapped with layer l's restore (norms) and fused
    GEMVs (matrices), against the same copies alone and the same ops alone."""
    import torch
    blob_host = []
    for seed_shift in (0, 1):
        ps = parts if seed_shift == 0 else build_layer(args.seed + 1, 0, "layer")
        size = sum(c.size for _, _, c, _ in ps)
        b = torch.empty(size, dtype=torch.uint8).pin_memory()
        o = 0
        for _, _, c, _ in ps:
            b.numpy()[o:o + c.size] = c
            o += c.size
        blob_host.append((b, ps))
    buf_bytes = max(b.numel() for b, _ in blob_host)
    bufs = [torch.empty(buf_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    compute, copy = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    out = {"layers": layers, "distinct_pinned_layers": len(blob_host),
           "layer_compressed_bytes": int(blob_host[0][0].numel())}
    for B in (1, 4):
        keep = []
        ops_per_blob = [_layer_ops(afx, ps, B, dev, keep) for _, ps in blob_host]
        seq = [(blob_host[l % 2][0], ops_per_blob[l % 2]) for l in range(layers)]
        copies_only = [(blob_host[l % 2][0], []) for l in range(layers)]

        def timed(layer_list):
            for _ in range(2):
                afx.afx_stream_run(layer_list, bufs, buf_bytes, compute, copy)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 3
            e0.record(compute)
            for _ in range(reps):
                afx.afx_stream_run(layer_list, bufs, buf_bytes, compute, copy)
            e1.record(compute)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        step_ms = timed(seq)
        copy_ms = timed(copies_only)
        # the same ops with every layer already on the device: no copies at all
        dev_blobs = [b.to(dev) for b, _ in blob_host]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(compute):
            e0.record(compute)
            for l in range(layers):
                ops = ops_per_blob[l % 2]
                i = 0
                while i < len(ops):
                    j = i + 1
                    while j < len(ops) and ops[j].kind == ops[i].kind:
                        j += 1
                    grp = ops[i:j]
                    conts = [dev_blobs[l % 2][op.offset:op.offset + op.desc.container_bytes] for op in grp]
                    if grp[0].kind == afx.AFX_OP_DECODE:
                        outs = [torch.empty(op.desc.n, dtype=torch.int16, device=dev) for op in grp]
                        afx.afx_decode_batch([op.desc for op in grp], conts, outs)
                    else:
                        import ctypes
                        arr = (afx.afx_desc * len(grp))(*[op.desc for op in grp])
                        ptrs = lambda xs: (ctypes.c_void_p * len(xs))(*xs)
                        st = afx._lib.afx_decode_gemv_batch(
                            arr, ptrs([c.data_ptr() for c in conts]), (ctypes.c_uint32 * len(grp))(*[op.rows for op in grp]),
                            (ctypes.c_uint32 * len(grp))(*[op.cols for op in grp]), ptrs([op.x_dev for op in grp]), B,
                            ptrs([op.out_dev for op in grp]), ptrs([op.workspace_dev for op in grp]),
                            (ctypes.c_uint64 * len(grp))(*[op.workspace_bytes for op in grp]), len(grp),
                            compute.cuda_stream, None)
                        assert st == 0
                    i = j
            e1.record(compute)
        torch.cuda.synchronize()
        compute_ms = e0.elapsed_time(e1)
        per_layer_copy = copy_ms / layers
        out[f"batch{B}"] = {"step_ms": step_ms, "copy_only_ms": copy_ms, "compute_only_ms": compute_ms,
                            "step_over_copy": step_ms / copy_ms,
                            "hidden": step_ms <= 1.05 * copy_ms + compute_ms / layers,
                            "h2d_gbs": layers * blob_host[0][0].numel() / (copy_ms * 1e-3) / 1e9,
                            "per_layer_copy_ms": per_layer_copy, "per_layer_compute_ms": compute_ms / layers}
        del keep
    return out


def run_cpu_baseline(parts):
    """The CPU oracle on the host's threads over as many of the workload's
    2^21-weight slices as divide evenly among them (every thread busy for
    the whole sample), and one slice on one thread."""
    threads = os.cpu_count() or 1
    slices = sum(w.size // ORACLE_SLICE for _, w, _, _ in parts)
    sample = oracle_sample(part_tensors(parts), threads * max(1, slices // threads))
    threads = max(1, min(threads, len(sample)))
    dt, nw = time_oracle(sample, threads)
    dt1, nw1 = time_oracle(sample[:1], 1)
    return {"value": elem_bytes(fmt_of(parts)) * nw / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(sample)} containers ({nw} weights) of the workload's "
                      f"{sum(w.size for _, w, _, _ in parts)}, {len(sample) // threads} per thread on {threads} threads",
            "weights_per_s": nw / dt, "one_core_weights_per_s": nw1 / dt1, "cpu": cpu_model()}


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
