"""The bounds-checked build (AFX_DEBUG_BOUNDS=1, libafx_debug.so) on the
restore path: across ragged sizes, the 12-bit-table path, long codes, host
containers, E4M3 and FP16 elements, partial state tables (escapes), the
fused GEMV and corrupt containers, with one chunk a lane and again with
two (sub-tiles decoded whole and in two halves), no range a kernel
touches ever leaves its buffer.  The check runs in a child process that
loads the debug library; compute-sanitizer is not available here."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np, torch
from weight_streaming_canonical_gb300 import build
build.build(debug_bounds=True)
from weight_streaming_canonical_gb300 import afx, synth
assert afx.DEBUG_BOUNDS
statuses = []

def restore(c, d, host=False):
    cont = torch.from_numpy(c).cuda() if not host else torch.from_numpy(c).pin_memory()
    e4m3 = d.format == afx.AFX_FMT_E4M3
    out = torch.empty(max(d.n, 1), dtype=torch.uint8 if e4m3 else torch.int16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode(d, cont, out[:d.n] if d.n else out, status_dev=st)
    torch.cuda.synchronize()
    got = out[:d.n].cpu().numpy()
    return (got if e4m3 else got.view(np.uint16)), int(st.item())

for n in (1, 1000, 65_537, 3_000_017):
    w = synth.normal(n, seed=n)
    got, st = restore(*afx.encode(w))
    statuses.append(("normal", n, st, bool(np.array_equal(got, w))))
w = synth.adversarial(1 << 20, seed=2)
got, st = restore(*afx.encode(w))
statuses.append(("adversarial", w.size, st, bool(np.array_equal(got, w))))
w = synth.all_bf16_patterns()
for T in (4, 32):
    got, st = restore(*afx.encode(w, chunk_bytes=T))
    statuses.append(("patterns", T, st, bool(np.array_equal(got, w))))
w = synth.normal(500_000, seed=5)
got, st = restore(*afx.encode(w), host=True)
statuses.append(("host", w.size, st, bool(np.array_equal(got, w))))
for n in (1, 17, 999_999):  # E4M3: raw nibbles, byte outputs
    w = synth.normal_e4m3(n, seed=n)
    got, st = restore(*afx.encode(w, fmt=afx.AFX_FMT_E4M3))
    statuses.append(("e4m3", n, st, bool(np.array_equal(got, w))))
w = synth.normal_e4m3(300_001, seed=8)
got, st = restore(*afx.encode(w, fmt=afx.AFX_FMT_E4M3), host=True)
statuses.append(("e4m3 host", w.size, st, bool(np.array_equal(got, w))))
w = synth.normal_fp16(300_001, seed=8)
got, st = restore(*afx.encode(w, fmt=afx.AFX_FMT_FP16))
statuses.append(("fp16", w.size, st, bool(np.array_equal(got, w))))
# a tree past the state table (rows for its shallowest nodes, escapes)
w = synth.exponent_mix(400_003, 90, ratio=0.9, seed=31)
cp, dp = afx.encode(w)
assert afx.afx_decode_table_kind(dp)[0] == afx.AFX_TABLE_PARTIAL
got, st = restore(cp, dp)
statuses.append(("partial", w.size, st, bool(np.array_equal(got, w))))
got, st = restore(cp, dp, host=True)
statuses.append(("partial host", w.size, st, bool(np.array_equal(got, w))))
bad = cp.copy()
bad[dp.off_exp: dp.off_exp + dp.n_chunks * dp.chunk_bytes] = np.random.default_rng(12).integers(
    0, 256, size=dp.n_chunks * dp.chunk_bytes, dtype=np.uint8)
statuses.append(("garbage partial", 0, restore(bad, dp)[1], None))
# corrupt containers: must be flagged, never read or write out of range
rng = np.random.default_rng(9)
w = synth.normal(400_000, seed=6)
c, d = afx.encode(w)
bad = c.copy()
bad[d.off_exp: d.off_exp + d.n_chunks * d.chunk_bytes] = rng.integers(0, 256, size=d.n_chunks * d.chunk_bytes,
                                                                        dtype=np.uint8)
statuses.append(("garbage stream", 0, restore(bad, d)[1], None))
bad = c.copy()
idx = d.off_chunk + 2 * rng.integers(0, d.n_chunks, size=64)
bad[idx] ^= np.uint8(0xA5)
statuses.append(("chunk index", 0, restore(bad, d)[1], None))
bad = c.copy()
bad[d.off_block + 8: d.off_block + 16] = 0xFF
statuses.append(("block index", 0, restore(bad, d)[1], None))
# the fused GEMV on the warp path
rows, cols = 96, 5120
W = synth.normal(rows * cols, seed=7)
c, d = afx.encode(W)
x = torch.from_numpy(synth.activations(2, cols, seed=1).view(np.int16)).cuda()
y = torch.empty((2, rows), dtype=torch.float32, device="cuda")
ws = torch.empty(afx.afx_decode_gemv_workspace(d, 2) // 4 + 4, dtype=torch.float32, device="cuda")
st = torch.zeros(1, dtype=torch.int32, device="cuda")
afx.afx_decode_gemv(d, torch.from_numpy(c).cuda(), rows, cols, x, y, ws, status_dev=st)
torch.cuda.synchronize()
statuses.append(("gemv", rows * cols, int(st.item()), None))
# the fused GEMV with a partial state table
W = synth.exponent_mix(rows * cols, 90, ratio=0.9, seed=8)
c, d = afx.encode(W)
y4 = torch.empty((4, rows), dtype=torch.float32, device="cuda")
x4 = torch.from_numpy(synth.activations(4, cols, seed=2).view(np.int16)).cuda()
ws = torch.empty(afx.afx_decode_gemv_workspace(d, 4) // 4 + 4, dtype=torch.float32, device="cuda")
st.zero_()
afx.afx_decode_gemv(d, torch.from_numpy(c).cuda(), rows, cols, x4, y4, ws, status_dev=st)
torch.cuda.synchronize()
statuses.append(("gemv partial", rows * cols, int(st.item()), None))
# randomized corruption: bytes of every section replaced, flipped or zeroed,
# in all three formats; the kernels must flag or restore, never leave a buffer
rng = np.random.default_rng(2026)
fuzz_flagged = fuzz_exact = 0
bases = [afx.encode(synth.normal(300_001, seed=21)), afx.encode(synth.normal_fp16(200_003, seed=22), fmt=1),
         afx.encode(synth.normal_e4m3(300_007, seed=23), fmt=2), afx.encode(synth.adversarial(1 << 18, seed=24)),
         afx.encode(synth.exponent_mix(200_003, 90, ratio=0.9, seed=25))]
for trial in range(150):
    c0, d = bases[trial % len(bases)]
    bad = c0.copy()
    section = trial % 4
    lo, hi = [(d.off_exp, d.off_exp + d.exp_bytes), (d.off_sm, d.off_chunk),
              (d.off_chunk, d.off_block), (d.off_block, d.container_bytes)][section]
    k = int(rng.integers(1, 64))
    idx = rng.integers(lo, hi, size=k)
    mode = trial % 3
    if mode == 0:
        bad[idx] = rng.integers(0, 256, size=k, dtype=np.uint8)
    elif mode == 1:
        bad[idx] ^= np.uint8(1) << rng.integers(0, 8, size=k).astype(np.uint8)
    else:
        bad[idx] = 0
    got, st = restore(bad, d)
    if st != 0:
        fuzz_flagged += 1
    else:
        fuzz_exact += 1
statuses.append(("fuzz", fuzz_flagged, 0, None))
statuses.append(("fuzz_clean", fuzz_exact, 0, None))
# the same kinds of case with two chunks a lane (64-chunk sub-tiles), forced
# on for these small tensors; cases are tagged "2:"
import os
os.environ["AFX_CHUNKS_A_LANE"] = "2"
c, d = afx.encode(synth.normal(1000, seed=3))
assert afx.afx_decode_chunks_a_lane([d], [torch.from_numpy(c).cuda()]) == [2]
for n in (1000, 3_000_017):
    w = synth.normal(n, seed=n + 1)
    got, st = restore(*afx.encode(w))
    statuses.append(("2:normal", n, st, bool(np.array_equal(got, w))))
w = synth.all_bf16_patterns()
for T in (4, 32):
    got, st = restore(*afx.encode(w, chunk_bytes=T))
    statuses.append(("2:patterns", T, st, bool(np.array_equal(got, w))))
w = synth.normal_e4m3(999_999, seed=4)
got, st = restore(*afx.encode(w, fmt=afx.AFX_FMT_E4M3))
statuses.append(("2:e4m3", w.size, st, bool(np.array_equal(got, w))))
w = synth.normal_fp16(300_001, seed=9)
got, st = restore(*afx.encode(w, fmt=afx.AFX_FMT_FP16))
statuses.append(("2:fp16", w.size, st, bool(np.array_equal(got, w))))
# sub-tiles that overflow the stage (decoded in two halves): a run of
# weights that all share the most common exponent, and 1-bit codes
a = synth.normal(1_500_007, seed=41)
top = np.bincount((a >> 7) & 0xFF, minlength=256).argmax()
mid = (np.random.default_rng(5).integers(0, 1 << 16, 65_536).astype(np.uint16) & 0x807F) | np.uint16(top << 7)
w = np.concatenate([a, mid, synth.normal(1_200_001, seed=42)])
got, st = restore(*afx.encode(w))
statuses.append(("2:halves", w.size, st, bool(np.array_equal(got, w))))
w = np.where(np.random.default_rng(6).random(1_000_001) < 0.6, 0x3F80, 0x3F00).astype(np.uint16)
got, st = restore(*afx.encode(w))
statuses.append(("2:one-bit", w.size, st, bool(np.array_equal(got, w))))
w = synth.normal(400_000, seed=16)
c, d = afx.encode(w)
bad = c.copy()
bad[d.off_exp: d.off_exp + d.n_chunks * d.chunk_bytes] = rng.integers(0, 256, size=d.n_chunks * d.chunk_bytes,
                                                                        dtype=np.uint8)
statuses.append(("2:garbage stream", 0, restore(bad, d)[1], None))
bad = c.copy()
idx = d.off_chunk + 2 * rng.integers(0, d.n_chunks, size=64)
bad[idx] ^= np.uint8(0xA5)
statuses.append(("2:chunk index", 0, restore(bad, d)[1], None))
bad = c.copy()
bad[d.off_block + 8: d.off_block + 16] = 0xFF
statuses.append(("2:block index", 0, restore(bad, d)[1], None))
# the batch-1 GEMV with two chunks a lane
rows, cols = 96, 5120
c, d = afx.encode(synth.normal(rows * cols, seed=17))
x1 = torch.from_numpy(synth.activations(1, cols, seed=3).view(np.int16)).cuda()
y1 = torch.empty((1, rows), dtype=torch.float32, device="cuda")
ws = torch.empty(afx.afx_decode_gemv_workspace(d, 1) // 4 + 4, dtype=torch.float32, device="cuda")
st = torch.zeros(1, dtype=torch.int32, device="cuda")
afx.afx_decode_gemv(d, torch.from_numpy(c).cuda(), rows, cols, x1, y1, ws, status_dev=st)
torch.cuda.synchronize()
statuses.append(("2:gemv", rows * cols, int(st.item()), None))
flagged = exact = 0
for trial in range(60):
    c0, d = bases[trial % 3]
    bad = c0.copy()
    lo, hi = [(d.off_exp, d.off_exp + d.exp_bytes), (d.off_sm, d.off_chunk),
              (d.off_chunk, d.off_block), (d.off_block, d.container_bytes)][trial % 4]
    k = int(rng.integers(1, 64))
    bad[rng.integers(lo, hi, size=k)] ^= np.uint8(1) << rng.integers(0, 8, size=k).astype(np.uint8)
    got, st = restore(bad, d)
    flagged += st != 0
    exact += st == 0
statuses.append(("2:fuzz", flagged, 0, None))
statuses.append(("2:fuzz_clean", exact, 0, None))
del os.environ["AFX_CHUNKS_A_LANE"]
bits, checked = afx.afx_debug_bounds_report()
print(json.dumps({"bits": bits, "checked": checked, "cases": statuses}))
"""


def test_bounds_checked_build_reports_no_violation():
    env = dict(os.environ, AFX_DEBUG_BOUNDS="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    rep = json.loads(r.stdout.strip().splitlines()[-1])
    assert rep["checked"]
    for tagged, size, status, exact in rep["cases"]:
        kind = tagged.split(":", 1)[-1]  # "2:" marks the cases with two chunks a lane
        if kind in ("garbage stream", "chunk index", "block index", "garbage partial"):
            assert status != 0, kind
        elif kind == "fuzz":
            assert size > 0  # corruptions the kernels flagged
        else:
            assert status == 0 and exact in (True, None), (kind, size)
    assert rep["bits"] == 0, f"bounds checks failed: {rep['bits']:#x}"


@pytest.mark.skipif(os.environ.get("AFX_DEBUG_BOUNDS", "0") == "1", reason="the session runs the checked build")
def test_regular_build_reports_nothing(afx):
    bits, checked = afx.afx_debug_bounds_report()
    assert bits == 0 and not checked
