"""GPU decode parity: afx_decode (through the C ABI) against the CPU oracle,
bit for bit, from tiny ragged inputs to the full workloads."""
import numpy as np
import pytest

import oracle
from afx_testutil import gpu_decode
from weight_streaming_canonical_gb300 import synth

pytestmark = pytest.mark.gpu


def _check(afx, w, chunk_bytes=0, **kw):
    w = np.ascontiguousarray(w).reshape(-1)
    c, d = afx.encode(w, chunk_bytes=chunk_bytes)
    ref, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(ref, w)
    out, status, intact = gpu_decode(afx, c, d, **kw)
    assert status == 0
    assert intact, "wrote outside the output range"
    mism = np.flatnonzero(out != ref)
    assert mism.size == 0, f"{mism.size} mismatches, first at {mism[:5]}"
    return c, d


@pytest.mark.parametrize("n", [1, 2, 7, 8, 9, 15, 16, 17, 255, 256, 257, 1000, 4095, 4097, 25_000, 65_537,
                               300_007, 1_000_003])
def test_ragged_sizes(afx, n):
    _check(afx, synth.normal(n, seed=n), out_pad=24)


@pytest.mark.parametrize("T", [4, 8, 16, 32])
def test_every_bf16_pattern_every_chunk_size(afx, T):
    w = synth.all_bf16_patterns()
    rng = np.random.default_rng(T)
    _check(afx, np.concatenate([w, rng.permutation(w), w[::-1]]), chunk_bytes=T)


@pytest.mark.parametrize("T", [4, 8, 16])
def test_byte_steps_every_chunk_size(afx, T):
    c, d = _check(afx, synth.normal(700_001, seed=T), chunk_bytes=T, out_pad=16)
    assert d.chunk_bytes == T


def test_byte_steps_with_32_byte_chunks(afx):
    # 16 nearly equally likely exponents: every code is 4 bits, so T = 32 is allowed
    c, d = _check(afx, synth.exponent_mix(600_011, 16, ratio=0.97, seed=2), out_pad=16)
    assert d.chunk_bytes == 32 and min(l for l in d.len if l) == 4


@pytest.mark.parametrize("nsym,ratio", [(51, 0.85), (52, 0.85), (57, 0.85), (58, 0.85), (80, 0.9), (120, 0.94),
                                        (200, 0.97)])
def test_largest_state_table_and_the_trees_past_it(afx, nsym, ratio):
    # with 32 warps staging 16-byte chunks, rows for 50 internal nodes fit:
    # 51 exponents decode with the whole state table, 52 to 80 with rows for
    # the 50 shallowest nodes and escapes at the others; 120 and 200 (32-byte
    # chunks, escapes in most chunks) with the 12-bit table
    c, d = _check(afx, synth.exponent_mix(3_000_017, nsym, ratio=ratio, seed=nsym), out_pad=16)
    assert d.nsym == nsym and min(l for l in d.len if l) >= 2
    expect = afx.AFX_TABLE_STATES if nsym <= 51 else afx.AFX_TABLE_PARTIAL if nsym <= 80 else afx.AFX_TABLE_LUT12
    assert afx.afx_decode_table_kind(d)[0] == expect


def test_table_kind_follows_the_tree(afx):
    def kind(w, fmt=0):
        return afx.afx_decode_table_kind(afx.encode(w, fmt=fmt)[1])
    fill = np.full(1000, 0x3F80, dtype=np.uint16)
    assert kind(fill) == (afx.AFX_TABLE_FILL, 0)
    assert kind(synth.exponent_mix(100_000, 2, ratio=0.5, seed=1))[0] == afx.AFX_TABLE_LUT12  # 1-bit codes
    normal = synth.normal(300_000, seed=1)
    assert kind(normal) == (afx.AFX_TABLE_STATES, afx.encode(normal)[1].nsym - 1)  # every internal node
    k51, rows = kind(synth.exponent_mix(3_000_017, 51, ratio=0.85, seed=51))
    assert k51 == afx.AFX_TABLE_STATES and rows == 50
    assert kind(synth.exponent_mix(3_000_017, 52, ratio=0.85, seed=52)) == (afx.AFX_TABLE_PARTIAL, rows)
    assert kind(synth.exponent_mix(2_000_003, 90, ratio=0.9, seed=9)) == (afx.AFX_TABLE_PARTIAL, rows)
    # a flat tree in 32-byte chunks: fewer rows fit and most codes pass a
    # node without one, so the 12-bit table is the faster decoder
    assert kind(synth.exponent_mix(1_500_007, 100, ratio=0.99, seed=3)) == (afx.AFX_TABLE_LUT12, 0)
    assert kind(synth.normal_fp16(100_000, seed=2), fmt=afx.AFX_FMT_FP16)[0] == afx.AFX_TABLE_STATES


@pytest.mark.parametrize("T", [4, 8])
def test_partial_state_tables_small_chunks(afx, T):
    # the escapes start at any bit of a chunk, also where a chunk is one word
    w = synth.exponent_mix(1_500_007, 100, ratio=0.92, seed=T)
    c, d = _check(afx, w, chunk_bytes=T, out_pad=16)
    assert d.chunk_bytes == T and afx.afx_decode_table_kind(d)[0] == afx.AFX_TABLE_PARTIAL


def test_partial_state_table_with_a_long_tail(afx):
    # the layer's distribution plus rare exponents across the whole range (the
    # shape of a checkpoint with outliers): 254 exponents, escapes are rare
    # and the rare codes are up to 19 bits long
    w = synth.long_tail(4_000_000, seed=5)
    c, d = _check(afx, w, out_pad=16)
    assert d.nsym > 60 and d.max_len > 16 and afx.afx_decode_table_kind(d)[0] == afx.AFX_TABLE_PARTIAL


def test_partial_state_tables_from_pinned_host_memory(afx):
    import torch
    w = synth.exponent_mix(2_000_003, 90, ratio=0.9, seed=9)
    c, d = afx.encode(w)
    assert afx.afx_decode_table_kind(d)[0] == afx.AFX_TABLE_PARTIAL
    out = torch.full((w.size,), 0x5A5A, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode(d, _pinned(c), out, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), w)


def test_batch_mixing_partial_and_whole_state_tables(afx):
    # wide trees go to launches of their own (70 exponents: a partial state
    # table; 130 exponents in 32-byte chunks: the 12-bit table); the batch's
    # outputs are all exact
    import torch
    ws = [synth.normal(700_001, seed=1), synth.exponent_mix(900_007, 70, ratio=0.9, seed=2),
          synth.exponent_mix(500_009, 30, ratio=0.8, seed=3), synth.exponent_mix(1_100_003, 130, ratio=0.95, seed=4),
          synth.adversarial(300_001, seed=5)]
    enc = [afx.encode(w) for w in ws]
    conts = [(_pinned(c) if i == 3 else torch.from_numpy(c).cuda()) for i, (c, _) in enumerate(enc)]
    outs = [torch.full((w.size,), 0x5A5A, dtype=torch.int16, device="cuda") for w in ws]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_batch([d for _, d in enc], conts, outs, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for w, o in zip(ws, outs):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), w)


def test_corrupt_stream_with_a_partial_state_table(afx):
    # flipped bits and a garbage stream: flagged (or, for a flip that still
    # decodes to the right count, a wrong tensor), never a hang or a write
    # outside the output
    w = synth.exponent_mix(600_011, 90, ratio=0.9, seed=12)
    c, d = afx.encode(w)
    assert afx.afx_decode_table_kind(d)[0] == afx.AFX_TABLE_PARTIAL
    rng = np.random.default_rng(4)
    for pos in rng.integers(0, d.total_bits // 8, size=8):
        bad = c.copy()
        bad[d.off_exp + int(pos)] ^= 0x10
        status, out = _decode_bad(afx, bad, d, w)
        assert status != 0 or not np.array_equal(out, w)
    bad = c.copy()
    bad[d.off_exp: d.off_exp + d.n_chunks * d.chunk_bytes] = rng.integers(
        0, 256, size=d.n_chunks * d.chunk_bytes, dtype=np.uint8)
    status, _ = _decode_bad(afx, bad, d, w)
    assert status != 0


def test_gaps_that_skip_zero_one_and_two_bytes(afx):
    # a chunk's first code may begin 0..23 bits in; 16 or more skips two bytes
    c, d = _check(afx, synth.exponent_mix(2_000_003, 50, ratio=0.75, seed=6))
    chunk = np.frombuffer(c[d.off_chunk: d.off_chunk + 2 * d.n_chunks].tobytes(), dtype="<u2")
    gaps = set(int(g) for g in np.unique(chunk & 31))
    assert gaps >= set(range(0, 17)) and min(l for l in d.len if l) == 2


@pytest.mark.parametrize("offset", [0, 8, 16, 24])
def test_output_offsets_keep_guards(afx, offset):
    _check(afx, synth.normal(123_457, seed=3), out_offset=offset, out_pad=16)


def test_single_exponent_tensor(afx):
    w = (np.full(100_003, 0x3F80, np.uint16) | (np.arange(100_003) % 128).astype(np.uint16)
         | ((np.arange(100_003) % 3 == 0).astype(np.uint16) << 15))
    c, d = _check(afx, w, out_pad=8)
    assert d.nsym == 1 and d.total_bits == 0


def test_two_exponent_tensor_uses_one_bit_codes(afx):
    w = np.where(np.random.default_rng(1).random(200_001) < 0.7, 0x3F80, 0x3F00).astype(np.uint16)
    c, d = _check(afx, w)
    assert d.chunk_bytes == 8 and d.total_bits == w.size


def test_norm_vector(afx):
    _check(afx, synth.layer_tensor("input_layernorm", seed=0))


def test_long_codes(afx):
    c, d = _check(afx, synth.adversarial(1 << 22, seed=1))
    assert d.max_len > 12  # exercises the second table level


def test_repeat_is_deterministic(afx):
    w = synth.normal(500_000, seed=9)
    c, d = afx.encode(w)
    a, s1, _ = gpu_decode(afx, c, d)
    b, s2, _ = gpu_decode(afx, c, d)
    assert s1 == s2 == 0 and np.array_equal(a, b) and np.array_equal(a, w)


def test_matrix_4096(afx):
    _check(afx, synth.matrix_4096(seed=0))


@pytest.mark.slow
def test_qwen3_layer_all_tensors(afx):
    for name, tensor in synth.layer(seed=0).items():
        _check(afx, tensor.reshape(-1))


@pytest.mark.slow
def test_adversarial_2_28(afx):
    w = synth.adversarial(1 << 28, seed=0)
    c, d = _check(afx, w)
    assert d.max_len == 24  # the 24-bit cap is exercised


# ---- corrupt input: status bits or a detected mismatch, never a hang ----------

def _decode_bad(afx, c, d, w):
    out, status, intact = gpu_decode(afx, c, d, out_pad=64)
    assert intact
    return status, out


def test_corrupt_chunk_index_is_flagged(afx):
    w = synth.normal(400_000, seed=11)
    c, d = afx.encode(w)
    for k in (0, 5, 300, d.n_chunks - 1):
        for flip in (1, 1 << 5, 1 << 9, 1 << 15):
            bad = c.copy()
            e = bad[d.off_chunk + 2 * k: d.off_chunk + 2 * k + 2].view(np.uint16)
            e[0] ^= flip
            status, out = _decode_bad(afx, bad, d, w)
            assert status != 0 or np.array_equal(out, w)


def test_corrupt_block_index_is_flagged(afx):
    w = synth.normal(400_000, seed=12)
    c, d = afx.encode(w)
    for b in range(d.n_blocks + 1):
        bad = c.copy()
        bad[d.off_block + 8 * b] ^= 0x3
        status, out = _decode_bad(afx, bad, d, w)
        assert status & afx.AFX_DEV_BAD_BLOCK


def test_corrupt_stream_is_detected(afx):
    w = synth.normal(400_000, seed=13)
    c, d = afx.encode(w)
    rng = np.random.default_rng(0)
    for pos in rng.integers(0, d.total_bits // 8, size=12):  # inside the coded bits, not the padding
        bad = c.copy()
        bad[d.off_exp + int(pos)] ^= 0x20
        status, out = _decode_bad(afx, bad, d, w)
        assert status != 0 or not np.array_equal(out, w)


def test_header_n_mismatch_is_flagged(afx):
    w = synth.normal(70_000, seed=5)
    c, d = afx.encode(w)
    bad = c.copy()
    bad[8] ^= 0x04  # n changes, section layout does not
    d2 = afx.afx_parse_header(bad)
    status, _ = _decode_bad(afx, bad, d2, w)
    assert status & afx.AFX_DEV_BAD_BLOCK


def test_garbage_stream_never_hangs(afx):
    w = synth.normal(300_000, seed=14)
    c, d = afx.encode(w)
    bad = c.copy()
    rng = np.random.default_rng(1)
    bad[d.off_exp: d.off_exp + d.n_chunks * d.chunk_bytes] = rng.integers(
        0, 256, size=d.n_chunks * d.chunk_bytes, dtype=np.uint8)
    status, _ = _decode_bad(afx, bad, d, w)
    assert status != 0


@pytest.mark.parametrize("n", [200_003, 3_000_017])
def test_staging_wait_that_runs_out_is_flagged_and_the_gpu_stays_usable(afx, n):
    # failure injection: the staging barriers are armed and no copy is issued,
    # so every warp's first wait gives up; nothing is left in flight
    import torch
    w = synth.normal(n, seed=31)
    c, d = afx.encode(w)
    dev = torch.from_numpy(c).cuda()
    out = torch.full((n,), 0x5A5A, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_test_restore_stalled(d, dev, out, 2000, status)
    torch.cuda.synchronize()
    assert status.item() & afx.AFX_DEV_TIMEOUT
    assert not status.item() & afx.AFX_DEV_UNDRAINED  # no copy was issued, so none is waited for
    assert bool((out == 0x5A5A).all())
    # the same context restores the tensor correctly afterwards
    got, st, _ = gpu_decode(afx, c, d)
    assert st == 0 and np.array_equal(got, w)


def test_stalled_restore_rejects_bad_arguments(afx):
    import torch
    c, d = afx.encode(synth.normal(10_000, seed=2))
    dev = torch.from_numpy(c).cuda()
    out = torch.empty(d.n, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for polls in (0, (1 << 22) + 1):
        with pytest.raises(afx.AfxError):
            afx.afx_test_restore_stalled(d, dev, out, polls, status)


def test_host_side_argument_errors(afx):
    import torch
    w = synth.normal(10_000, seed=15)
    c, d = afx.encode(w)
    dev = torch.from_numpy(c).cuda()
    out = torch.empty(d.n + 8, dtype=torch.int16, device="cuda")
    with pytest.raises(afx.AfxError):
        afx.afx_decode(d, dev, out[1:])  # output not 16-byte aligned
    with pytest.raises(afx.AfxError):
        afx.afx_decode(d, dev[1:], out)  # container not 16-byte aligned
    d_bad = afx.afx_parse_header(c)
    d_bad.off_sm += 256
    with pytest.raises(afx.AfxError):
        afx.afx_decode(d_bad, dev, out)
    c32 = oracle.encode(w, np.array(afx.afx_build_code(w).len[:], np.uint8), 8, 32)
    d32 = afx.afx_parse_header(c32)
    with pytest.raises(afx.AfxError):  # the decoder runs 512 chunks per block
        afx.afx_decode(d32, torch.from_numpy(c32).cuda(), out)


# ---- several containers in one launch ------------------------------------------

def test_batch_of_mixed_tensors_in_one_launch(afx):
    import torch
    tensors = [synth.normal(1_000_003, seed=1), synth.layer_tensor("input_layernorm", seed=2),
               np.full(4099, 0x3F80, np.uint16), synth.adversarial(300_001, seed=3), synth.normal(7, seed=4),
               np.zeros(0, np.uint16), synth.normal(2_000_000, 1.0, 0.05, seed=5)]
    encoded = [afx.encode(w) for w in tensors]
    devs = [torch.from_numpy(c).cuda() for c, _ in encoded]
    outs = [torch.full((max(1, w.size),), 0x5A5A, dtype=torch.int16, device="cuda") for w in tensors]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_batch([d for _, d in encoded], devs, outs, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for w, o in zip(tensors, outs):
        got = o.cpu().numpy().view(np.uint16)
        assert np.array_equal(got[:w.size], w)


def test_the_next_kernel_on_the_stream_sees_every_output(afx):
    # a call of several launches (the ones after the first may start while
    # the one before it finishes): work queued on the same stream right
    # after it, with no synchronisation between, reads finished outputs
    import torch
    ws = [synth.normal(1_000_003 + 1001 * i, seed=300 + i) for i in range(40)]
    enc = [afx.encode(w) for w in ws]
    conts = [torch.from_numpy(c).cuda() for c, _ in enc]
    refs = [torch.from_numpy(w.view(np.int16)).cuda() for w in ws]
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    for rep in range(3):
        outs = [torch.full((w.size,), 0x5A5A, dtype=torch.int16, device="cuda") for w in ws]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            afx.afx_decode_batch([d for _, d in enc], conts, outs, stream=stream, status_dev=status)
            # compared on the device, on the same stream, before any host synchronisation
            flags = torch.stack([(o == r).all() for o, r in zip(outs, refs)])
        torch.cuda.synchronize()
        assert status.item() == 0 and bool(flags.all()), rep


def test_batch_longer_than_one_launch(afx):
    import torch
    tensors = [synth.normal(50_000 + 37 * i, seed=100 + i) for i in range(37)]  # more than 16 per launch
    encoded = [afx.encode(w) for w in tensors]
    devs = [torch.from_numpy(c).cuda() for c, _ in encoded]
    outs = [torch.empty(w.size, dtype=torch.int16, device="cuda") for w in tensors]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_batch([d for _, d in encoded], devs, outs, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for w, o in zip(tensors, outs):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), w)


@pytest.mark.slow
def test_qwen3_layer_in_one_launch(afx):
    import torch
    layer = synth.layer(seed=0)
    encoded = [afx.encode(t.reshape(-1)) for t in layer.values()]
    devs = [torch.from_numpy(c).cuda() for c, _ in encoded]
    outs = [torch.empty(d.n, dtype=torch.int16, device="cuda") for _, d in encoded]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_batch([d for _, d in encoded], devs, outs, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for (c, _), o in zip(encoded, outs):
        ref, st = oracle.decode(c)
        assert st == oracle.OK and np.array_equal(o.cpu().numpy().view(np.uint16), ref)


@pytest.mark.parametrize("n", [3_000_017, 9_000_001])
def test_sizes_where_a_cta_owns_several_blocks(afx, n):
    # more blocks than resident CTAs: every warp restores several sub-tiles in a row
    _check(afx, synth.normal(n, seed=n))


@pytest.mark.slow
def test_full_model_resident_bit_exact(afx):
    """All 362 tensors of the Qwen3-14B-shaped model (14.77B weights) resident
    on one GPU and restored by batched launches; every restored tensor equals
    its original bit for bit (compared on the device); the oracle decodes one
    sampled tensor of every kind as well."""
    import torch
    import bench
    parts = bench.build_layer(0, 0, "model")
    assert sum(d.n for _, _, _, d in parts) == synth.model_weight_count()
    conts = [torch.from_numpy(c).cuda() for _, _, c, _ in parts]
    outs = [torch.empty(d.n, dtype=torch.int16, device="cuda") for _, _, _, d in parts]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_batch([d for *_, d in parts], conts, outs, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for (name, w, _, _), o in zip(parts, outs):
        assert torch.equal(o, torch.from_numpy(w.reshape(-1).view(np.int16)).cuda()), name
    sampled = {"embed_tokens", "layers.17.q_proj", "layers.39.input_layernorm", "lm_head"}
    for (name, w, c, _), o in zip(parts, outs):
        if name in sampled:
            ref, st = oracle.decode(c)
            assert st == oracle.OK and np.array_equal(o.cpu().numpy().view(np.uint16), ref), name


# ---- containers in pinned host memory (read by the kernel over the host link) ----

def _pinned(a: np.ndarray):
    import torch
    t = torch.empty(a.nbytes, dtype=torch.uint8).pin_memory()
    t.numpy()[:] = a.view(np.uint8).reshape(-1)
    return t


@pytest.mark.parametrize("n", [1, 1000, 65_537, 3_000_017])
@pytest.mark.parametrize("out_on_host", [False, True])
def test_restore_from_pinned_host_container(afx, n, out_on_host):
    import torch
    w = synth.normal(n, seed=50 + n)
    c, d = afx.encode(w)
    host_c = _pinned(c)
    if out_on_host:
        out = torch.full((n,), 0x5A5A, dtype=torch.int16).pin_memory()
    else:
        out = torch.full((n,), 0x5A5A, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode(d, host_c, out, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), w)


def test_batch_mixing_host_and_device_containers(afx):
    import torch
    ws = [synth.normal(200_000 + 7 * i, seed=60 + i) for i in range(4)] + [synth.adversarial(300_001, seed=3)]
    enc = [afx.encode(w) for w in ws]
    conts = [(_pinned(c) if i % 2 else torch.from_numpy(c).cuda()) for i, (c, _) in enumerate(enc)]
    outs = [torch.empty(w.size, dtype=torch.int16, device="cuda") for w in ws]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_batch([d for _, d in enc], conts, outs, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for w, o in zip(ws, outs):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), w)


def test_corrupt_host_container_is_flagged(afx):
    import torch
    w = synth.normal(500_000, seed=70)
    c, d = afx.encode(w)
    bad = c.copy()
    rng = np.random.default_rng(3)
    bad[d.off_exp: d.off_exp + d.n_chunks * d.chunk_bytes] = rng.integers(
        0, 256, size=d.n_chunks * d.chunk_bytes, dtype=np.uint8)
    out = torch.empty(d.n, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode(d, _pinned(bad), out, status_dev=status)
    torch.cuda.synchronize()
    assert status.item() != 0


def test_gemv_refuses_a_host_container(afx):
    import torch
    rows, cols = 64, 5120
    c, d = afx.encode(synth.normal(rows * cols, seed=71))
    x = torch.zeros((1, cols), dtype=torch.int16, device="cuda")
    y = torch.zeros((1, rows), dtype=torch.float32, device="cuda")
    ws = torch.empty(afx.afx_decode_gemv_workspace(d, 1) // 4 + 4, dtype=torch.float32, device="cuda")
    with pytest.raises((afx.AfxError, ValueError)):
        afx.afx_decode_gemv(d, _pinned(c), rows, cols, x, y, ws)


def test_block_index_entries_near_2_64_write_nothing_outside(afx):
    # a block-index entry of 2^64 - 1 makes start + count wrap back below n;
    # the restore must flag it and write nothing outside the output (the
    # guard elements on both sides stay as they were)
    w = synth.normal(400_003, seed=77)
    c, d = afx.encode(w)
    assert d.n_blocks > 4
    bad = c.copy()
    for b in range(1, int(d.n_blocks)):
        bad[d.off_block + 8 * b: d.off_block + 8 * b + 8] = 0xFF
    out, status, intact = gpu_decode(afx, bad, d, out_pad=64, out_offset=64)
    assert status & afx.AFX_DEV_BAD_BLOCK
    assert intact, "wrote outside the output range"
