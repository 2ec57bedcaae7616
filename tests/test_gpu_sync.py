"""afx_sync: the bounded host wait and the status read-back.  The timeout
case waits on a stream kept busy by a kernel that ends by itself (a timed
spin of a fraction of a second), so nothing ever hangs."""
import numpy as np
import pytest

from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu


def test_sync_ok_after_a_restore(afx):
    import torch
    w = synth.normal(300_001, seed=1)
    c, d = afx.encode(w)
    out = torch.empty(w.size, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        afx.afx_decode(d, torch.from_numpy(c).cuda(), out, stream=s, status_dev=status)
    st, word = afx.afx_sync(s, 10_000, status)
    assert (st, word) == (afx.AFX_OK, 0)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), w)


def test_sync_times_out_on_a_busy_stream_then_completes(afx):
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(4e8))  # a few hundred ms of GPU spin that ends by itself
    st, word = afx.afx_sync(s, 5)
    assert st == afx.AFX_E_TIMEOUT and word == 0
    st, word = afx.afx_sync(s, 0)  # no limit: waits for the spin to end
    assert st == afx.AFX_OK


def test_sync_reports_a_corrupt_container(afx):
    import torch
    w = synth.normal(400_000, seed=2)
    c, d = afx.encode(w)
    bad = c.copy()
    bad[d.off_chunk: d.off_chunk + 2 * d.n_chunks] = 0xFF  # every chunk index entry wrong
    out = torch.empty(w.size, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        afx.afx_decode(d, torch.from_numpy(bad).cuda(), out, stream=s, status_dev=status)
    st, word = afx.afx_sync(s, 10_000, status)
    assert st == afx.AFX_E_CORRUPT and word != 0


def test_sync_reads_a_pinned_host_status_word(afx):
    import torch
    w = synth.normal(50_000, seed=3)
    c, d = afx.encode(w)
    out = torch.empty(w.size, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32).pin_memory()
    afx.afx_decode(d, torch.from_numpy(c).cuda(), out, status_dev=torch.zeros(1, dtype=torch.int32, device="cuda"))
    st, word = afx.afx_sync(None, 10_000, status)
    assert (st, word) == (afx.AFX_OK, 0)
