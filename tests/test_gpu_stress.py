"""Randomized restores on three streams at once: batches of 1 to 6 tensors
drawn from a pool of sizes, distributions and element formats, every
restored tensor compared with its source bit for bit, for a fixed time,
with the launches' own choice of chunks a lane and with two forced."""
import time

import numpy as np
import pytest

from weight_streaming_canonical_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SECONDS = 15.0


def _pool(afx, dev, rng):
    import torch
    pool = []
    for i in range(30):
        kind = int(rng.integers(0, 6))
        n = int(rng.choice([0, 1, 7, 4099, 65536, 1_000_003, 5_000_000]))
        if kind == 0:
            w, fmt = synth.normal(n, seed=i), afx.AFX_FMT_BF16
        elif kind == 1:
            w, fmt = synth.normal(n, 1.0, 0.05, seed=i), afx.AFX_FMT_BF16
        elif kind == 2:
            w, fmt = synth.adversarial(max(n, 1), seed=i)[:n], afx.AFX_FMT_BF16
        elif kind == 3:
            w, fmt = np.full(n, 0x3F80, np.uint16) | (np.arange(n) % 128).astype(np.uint16), afx.AFX_FMT_BF16
        elif kind == 4:
            w, fmt = synth.normal_fp16(n, seed=i), afx.AFX_FMT_FP16
        else:
            w, fmt = synth.normal_e4m3(n, seed=i), afx.AFX_FMT_E4M3
        w = np.ascontiguousarray(w)
        c, d = afx.encode(w, fmt=fmt)
        pool.append((w, torch.from_numpy(c).to(dev), d, fmt))
    return pool


@pytest.mark.parametrize("lanes", ["auto", "2"])
def test_random_batches_on_three_streams_stay_bit_exact(afx, lanes, monkeypatch):
    # "2": every launch with two chunks a lane (forced; these tensors are
    # too small to take it by themselves)
    import torch
    if lanes != "auto":
        monkeypatch.setenv("AFX_CHUNKS_A_LANE", lanes)
    rng = np.random.default_rng(12345)
    dev = torch.device("cuda:0")
    pool = _pool(afx, dev, rng)
    streams = [torch.cuda.Stream() for _ in range(3)]
    launches = checks = 0
    failures = []
    t_end = time.time() + SECONDS
    while time.time() < t_end:
        pending = []
        for s in streams:
            idx = rng.choice(len(pool), size=int(rng.integers(1, 7)), replace=False)
            fmt = pool[idx[0]][3]
            items = [pool[i] for i in idx if pool[i][3] == fmt]  # one element format per launch
            e4m3 = fmt == afx.AFX_FMT_E4M3
            outs = [torch.empty(max(w.size, 1), dtype=torch.uint8 if e4m3 else torch.int16, device=dev)
                    for w, _, _, _ in items]
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            s.wait_stream(torch.cuda.current_stream())  # the zeroed status word and the outputs first
            afx.afx_decode_batch([d for _, _, d, _ in items], [c for _, c, _, _ in items], outs, stream=s,
                                 status_dev=st)
            launches += 1
            pending.append((items, outs, st))
        torch.cuda.synchronize()
        for items, outs, st in pending:
            if st.item() != 0:
                failures.append(("status", st.item()))
                continue
            for (w, _, _, fmt), o in zip(items, outs):
                got = o.cpu().numpy()
                if fmt != afx.AFX_FMT_E4M3:
                    got = got.view(np.uint16)
                checks += 1
                if not np.array_equal(got[:w.size], w):
                    failures.append(("mismatch", w.size, fmt))
    assert launches > 100 and checks > launches
    assert not failures, failures[:5]
