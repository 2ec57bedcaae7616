"""Host calls from several threads at once (ctypes releases the GIL, so the
library runs them concurrently): each thread encodes its own tensors and
restores them on its own stream, through the per-device caches the library
guards with a mutex.  Every result is bit-exact."""
import threading

import numpy as np
import pytest

from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu


def test_concurrent_encode_and_restore_on_separate_streams(afx):
    import torch
    errors, results = [], {}

    def work(k):
        try:
            s = torch.cuda.Stream()
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            for it in range(6):
                n = 200_003 + 40_009 * k + 13 * it
                fmt = (k + it) % 3
                w = (synth.normal(n, seed=k * 100 + it) if fmt == 0 else synth.normal_fp16(n, seed=k * 100 + it)
                     if fmt == 1 else synth.normal_e4m3(n, seed=k * 100 + it))
                c, d = afx.encode(w, fmt=fmt)
                out = torch.empty(n, dtype=torch.uint8 if fmt == 2 else torch.int16, device="cuda")
                with torch.cuda.stream(s):
                    afx.afx_decode(d, torch.from_numpy(c).to("cuda", non_blocking=False), out, stream=s,
                                   status_dev=status)
                st, word = afx.afx_sync(s, 30_000, status)
                got = out.cpu().numpy()
                results[(k, it)] = st == afx.AFX_OK and word == 0 and np.array_equal(
                    got if fmt == 2 else got.view(np.uint16), w)
        except Exception as e:  # reported below, on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not errors, errors
    assert len(results) == 24 and all(results.values()), results
