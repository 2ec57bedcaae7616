"""The restore with two chunks a lane (64-chunk sub-tiles, one span of 2T
stream bytes a lane), forced on with AFX_CHUNKS_A_LANE=2 so that small and
ragged tensors take it too: the decode parity, pattern, format, GEMV and
corruption tests run again that way against the CPU oracle, plus the
sub-tiles whose codes overflow the stage (decoded in two halves).
Large launches take this path by themselves; these tests reach it at every
size."""
import numpy as np
import pytest

import oracle
from afx_testutil import gpu_decode, gpu_gemv, within_gemv_tolerance
from weight_streaming_canonical_gb300 import synth

from test_gpu_decode import (  # noqa: F401  (collected again here, with two chunks a lane)
    test_ragged_sizes, test_every_bf16_pattern_every_chunk_size, test_byte_steps_every_chunk_size,
    test_byte_steps_with_32_byte_chunks, test_gaps_that_skip_zero_one_and_two_bytes,
    test_output_offsets_keep_guards, test_two_exponent_tensor_uses_one_bit_codes, test_norm_vector,
    test_long_codes, test_repeat_is_deterministic, test_matrix_4096, test_corrupt_chunk_index_is_flagged,
    test_corrupt_block_index_is_flagged, test_corrupt_stream_is_detected, test_header_n_mismatch_is_flagged,
    test_garbage_stream_never_hangs, test_staging_wait_that_runs_out_is_flagged_and_the_gpu_stays_usable,
    test_batch_of_mixed_tensors_in_one_launch, test_batch_longer_than_one_launch,
    test_sizes_where_a_cta_owns_several_blocks, test_block_index_entries_near_2_64_write_nothing_outside)
from test_gpu_gemv import (  # noqa: F401
    test_shapes_and_batches, test_corrupt_stream_is_flagged_by_the_gemv, test_unit_vector_gives_a_column_exactly,
    test_unit_vector_per_batch_row_gives_its_own_column_exactly, test_zero_activation_gives_zero,
    test_reproducible_bit_for_bit, test_row_longer_than_a_block, test_gemv_batch_of_products_in_one_launch)
from test_gpu_formats import (  # noqa: F401
    test_e4m3_ragged_sizes, test_fp16_ragged_sizes, test_e4m3_every_pattern_every_chunk_size,
    test_fp16_every_pattern, test_e4m3_byte_step_path_and_12_bit_path, test_mixed_format_batch,
    test_e4m3_corrupt_stream_is_flagged, test_fp16_small_chunks_ragged, test_fp16_every_hi_pattern_at_every_position)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def two_chunks_a_lane(monkeypatch):
    monkeypatch.setenv("AFX_CHUNKS_A_LANE", "2")


def _check(afx, w, **kw):
    c, d = afx.encode(w)
    ref, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(ref, w)
    out, status, intact = gpu_decode(afx, c, d, **kw)
    assert status == 0 and intact
    mism = np.flatnonzero(out != ref)
    assert mism.size == 0, f"{mism.size} mismatches, first at {mism[:5]}"
    return c, d


@pytest.mark.parametrize("run", [3000, 65_536, 150_001])
def test_sub_tiles_that_overflow_the_stage(afx, run):
    # a run of weights that all share the most common exponent codes to 2
    # bits a weight: 4096 codes in a 64-chunk sub-tile, more than the stage
    # holds, so those sub-tiles (and the ones where the run begins and ends)
    # are decoded in two halves between sub-tiles decoded whole
    a = synth.normal(1_500_007, seed=41)
    b = synth.normal(1_200_001, seed=42)
    top = np.bincount((a >> 7) & 0xFF, minlength=256).argmax()
    mid = (np.random.default_rng(run).integers(0, 1 << 16, run).astype(np.uint16) & 0x807F) | np.uint16(top << 7)
    w = np.concatenate([a, mid, b])
    c, d = _check(afx, w, out_pad=16)
    assert min(l for l in d.len if l) == 2


def test_one_bit_codes_every_sub_tile_in_halves(afx):
    # two exponents: 1-bit codes, 64 codes a 8-byte chunk, every sub-tile
    # overflows; the 12-bit table decodes them
    w = np.where(np.random.default_rng(5).random(3_000_001) < 0.6, 0x3F80, 0x3F00).astype(np.uint16)
    w |= (np.arange(w.size) % 251).astype(np.uint16) & 0x807F
    c, d = _check(afx, w, out_pad=8)
    assert d.chunk_bytes == 8


def test_the_forced_launches_take_two_chunks_a_lane(afx, monkeypatch):
    import torch
    ws = [(synth.normal(1000, seed=1), 0), (synth.all_bf16_patterns(), 0), (synth.normal_e4m3(300_007, seed=2), 2),
          (synth.normal_fp16(200_003, seed=3), 1), (np.full(4099, 0x3F80, np.uint16), 0)]
    enc = [afx.encode(w, fmt=f) for w, f in ws]
    devs = [torch.from_numpy(c).cuda() for c, _ in enc]
    assert afx.afx_decode_chunks_a_lane([d for _, d in enc], devs) == [2, 2, 2, 2, 0]
    host = [torch.from_numpy(enc[0][0]).pin_memory()]
    assert afx.afx_decode_chunks_a_lane([enc[0][1]], host) == [1]  # host containers: one chunk a lane
    monkeypatch.setenv("AFX_CHUNKS_A_LANE", "1")
    assert afx.afx_decode_chunks_a_lane([d for _, d in enc], devs) == [1, 1, 1, 1, 0]
    monkeypatch.delenv("AFX_CHUNKS_A_LANE")
    assert afx.afx_decode_chunks_a_lane([d for _, d in enc], devs) == [1, 1, 1, 1, 0]  # too small to pay


def test_a_layer_takes_two_chunks_a_lane_by_itself(afx, monkeypatch):
    # the layer's launch: 86 blocks a CTA, and its largest tree (28 nodes)
    # leaves a 3520-byte stage for about 3160 codes a sub-tile
    import torch
    monkeypatch.delenv("AFX_CHUNKS_A_LANE")
    enc = [afx.encode(t.reshape(-1)) for t in synth.layer(seed=0).values()]
    devs = [torch.from_numpy(c).cuda() for c, _ in enc]
    assert afx.afx_decode_chunks_a_lane([d for _, d in enc], devs) == [2] * len(enc)
    # and the matrix alone is 4.4 blocks a CTA: one chunk a lane
    c, d = afx.encode(synth.matrix_4096(seed=0))
    assert afx.afx_decode_chunks_a_lane([d], [torch.from_numpy(c).cuda()]) == [1]


def _overflow_matrix(run, cols):
    a = synth.normal(1_500_007, seed=41)
    b = synth.normal(1_200_001, seed=42)
    top = np.bincount((a >> 7) & 0xFF, minlength=256).argmax()
    mid = (np.random.default_rng(run).integers(0, 1 << 16, run).astype(np.uint16) & 0x807F) | np.uint16(top << 7)
    w = np.concatenate([a, mid, b])
    rows = w.size // cols
    return w[:rows * cols].reshape(rows, cols)


@pytest.mark.parametrize("B", [1, 4])
@pytest.mark.parametrize("cols", [4096, 8192])
def test_gemv_with_sub_tiles_in_halves(afx, B, cols):
    # the GEMV's workspace slots 2s and 2s + 1 hold the two halves of a
    # sub-tile that overflows the stage, and an empty slot after one merged
    # whole; the row fix-up adds them in order
    W = _overflow_matrix(65_536, cols)
    x = synth.activations(B, cols, seed=cols + B)
    rows = W.shape[0]
    c, d = afx.encode(W.reshape(-1))
    Wd, st = oracle.decode(c)
    assert st == oracle.OK
    y_ref, A = oracle.gemv(Wd.reshape(rows, cols), x)
    y, status = gpu_gemv(afx, c, d, rows, cols, x)
    assert status == 0 and not np.isnan(y).any()
    assert within_gemv_tolerance(y, y_ref, A)
