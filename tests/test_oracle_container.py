"""Pins for the oracle's container encode and bit-serial decode.

The hand-derived golden containers fix the bit order, the canonical order,
the chunk-index and block-index semantics and every header field.  The
exhaustive and brute-force round trips fix losslessness over every BF16
bit pattern (zeros, subnormals, infinities, NaN payloads).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from weight_streaming_canonical_gb300 import synth


def _u64(c, off):
    return int(np.frombuffer(c[off:off + 8].tobytes(), "<u8")[0])


def _u32(c, off):
    return int(np.frombuffer(c[off:off + 4].tobytes(), "<u4")[0])


def _u16(c, off):
    return int(np.frombuffer(c[off:off + 2].tobytes(), "<u2")[0])


HEADER_FIELDS = {  # name: (offset, bytes)
    "n": (8, 8), "total_bits": (16, 8), "T": (24, 4), "C": (28, 4), "n_chunks": (32, 8),
    "n_blocks": (40, 8), "off_exp": (48, 8), "exp_bytes": (56, 8), "off_sm": (64, 8),
    "off_chunk": (72, 8), "off_block": (80, 8), "container_bytes": (88, 8), "longest": (96, 4),
    "nsym": (100, 4), "fill": (104, 4),
}


def _field(c, name):
    off, nb = HEADER_FIELDS[name]
    return int.from_bytes(c[off:off + nb].tobytes(), "little")


def _lengths_from(d):
    lens = np.zeros(256, np.uint8)
    for k, v in d.items():
        lens[int(k)] = v
    return lens


def test_golden_tiny_container(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "container_tiny.json")))
    w = np.array([int(h, 16) for h in g["weights_hex"]], np.uint16)
    # the fixture's exponents and sign|mantissa bytes are the BF16 fields
    assert [int(e) for e in g["exponents"]] == [(int(x) >> 7) & 0xFF for x in w]
    lens = _lengths_from(g["lengths"])
    c = oracle.encode(w, lens, g["T"], g["C"])
    assert c.size == g["header"]["container_bytes"]
    assert _u32(c, 0) == 0x31584641 and _u16(c, 4) == 1 and _u16(c, 6) == 512
    for k, v in g["header"].items():
        assert _field(c, k) == v, k
    assert [int(c[256 + s]) for s in range(256)] == lens.tolist()
    assert not c[108:256].any()
    off_exp = g["header"]["off_exp"]
    words = [_u32(c, off_exp + 4 * i) for i in range(len(g["stream_words_hex"]))]
    assert words == [int(h, 16) for h in g["stream_words_hex"]]
    assert not c[off_exp + 4 * len(words): off_exp + g["header"]["exp_bytes"]].any()
    sm = c[g["header"]["off_sm"]: g["header"]["off_sm"] + w.size]
    assert sm.tolist() == [int(h, 16) for h in g["sm_hex"]]
    entries = [_u16(c, g["header"]["off_chunk"] + 2 * i) for i in range(g["header"]["n_chunks"])]
    assert entries == g["chunk_entries"]
    blocks = [_u64(c, g["header"]["off_block"] + 8 * i) for i in range(g["header"]["n_blocks"] + 1)]
    assert blocks == g["block_index"]
    out, st = oracle.decode(c)
    assert st == oracle.OK
    assert out.tolist() == w.tolist()


def test_golden_single_exponent_container(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "container_single_exponent.json")))
    w = np.array([int(h, 16) for h in g["weights_hex"]], np.uint16)
    lens = oracle.code_lengths(oracle.histogram(w))
    assert lens.max() == 0
    c = oracle.encode(w, lens, g["T"], g["C"])
    for k, v in g["header"].items():
        assert _field(c, k) == v, k
    sm = c[g["header"]["off_sm"]: g["header"]["off_sm"] + w.size]
    assert sm.tolist() == [int(h, 16) for h in g["sm_hex"]]
    assert _u64(c, g["header"]["off_block"]) == 5
    out, st = oracle.decode(c)
    assert st == oracle.OK and out.tolist() == w.tolist()


def _roundtrip(w, T=32, C=256, max_len=24):
    lens = oracle.code_lengths(oracle.histogram(w), max_len)
    c = oracle.encode(w, lens, T, C)
    out, st = oracle.decode(c)
    assert st == oracle.OK
    assert np.array_equal(out, w)
    return c


@pytest.mark.parametrize("T", [4, 8, 16, 32, 64])
def test_exhaustive_all_bf16_patterns(T):
    w = synth.all_bf16_patterns()
    _roundtrip(w, T=T, C=32 if T == 4 else 256)


def test_exhaustive_shuffled_and_repeated():
    rng = np.random.default_rng(5)
    base = synth.all_bf16_patterns()
    w = np.concatenate([rng.permutation(base), base[::-1], rng.permutation(base)])
    _roundtrip(w)
    _roundtrip(w[: (1 << 17) - 3], T=16, C=64)


def test_special_values_survive():
    specials = np.array([0x0000, 0x8000, 0x0001, 0x807F, 0x7F80, 0xFF80, 0x7FC0, 0x7F81, 0xFFFF,
                         0x7F7F, 0x0080, 0x3F80], np.uint16)
    w = np.tile(specials, 50)
    _roundtrip(w, T=4, C=32)


def test_brute_force_tiny_tensors():
    alphabet = [0x0000, 0x8000, 0x3F80, 0xBF80, 0x7FC1, 0x0003]
    for n in range(0, 4):
        for combo in itertools.product(alphabet, repeat=n):
            w = np.array(combo, np.uint16)
            for T, C in ((4, 32), (32, 256)):
                _roundtrip(w, T, C)


@pytest.mark.parametrize("n", [0, 1, 2, 7, 8, 9, 255, 256, 257, 1000, 4095, 4097, 65537])
def test_ragged_sizes(n):
    w = synth.normal(n, seed=n)
    for T, C in ((4, 32), (8, 64), (32, 256)):
        _roundtrip(w, T, C)


def test_two_symbol_tensor():
    w = np.array([0x3F80, 0x3F00] * 500 + [0x3F80], np.uint16)
    c = _roundtrip(w)
    assert _field(c, "total_bits") == w.size  # two symbols: one bit each


def test_chunk_gaps_cover_all_offsets():
    # long codes straddling chunk boundaries give many different offsets
    w = synth.adversarial(1 << 16, seed=3)
    c = _roundtrip(w, T=4, C=32, max_len=24)
    nch = _field(c, "n_chunks")
    off = _field(c, "off_chunk")
    gaps = {_u16(c, off + 2 * i) & 31 for i in range(nch)}
    assert len(gaps) >= 8


def test_adversarial_recipe_exceeds_24_bits_uncapped_and_cap_holds():
    import heapq
    # 2**26 draws of the full 2**28 recipe already need 26-bit codes uncapped
    w = synth.adversarial(1 << 26, seed=0)
    h = oracle.histogram(w)
    counts = [int(x) for x in h if x > 0]
    heap = [(c, 0) for c in counts]
    heapq.heapify(heap)
    while len(heap) > 1:
        a = heapq.heappop(heap)
        b = heapq.heappop(heap)
        heapq.heappush(heap, (a[0] + b[0], max(a[1], b[1]) + 1))
    assert heap[0][1] > 24  # unconstrained Huffman would need more than 24 bits
    lens = oracle.code_lengths(h, 24)
    assert int(lens.max()) == 24
    assert sum(1 << (24 - int(l)) for l in lens if l) == 1 << 24


def test_compressed_size_near_entropy_bound():
    w = synth.normal(1 << 21, seed=11)
    h = oracle.histogram(w).astype(np.float64)
    p = h[h > 0] / h.sum()
    H = float(-(p * np.log2(p)).sum())
    lens = oracle.code_lengths(oracle.histogram(w))
    c = oracle.encode(w, lens)
    total_bits = _field(c, "total_bits")
    n = w.size
    assert H * n <= total_bits < (H + 1) * n
    index_bytes = 2 * _field(c, "n_chunks") + 8 * (_field(c, "n_blocks") + 1)
    bound = n * (8 + H) / 8 + index_bytes + 512
    assert c.size <= 1.01 * bound


def _encoded(w):
    lens = oracle.code_lengths(oracle.histogram(w))
    return oracle.encode(w, lens, 8, 32)


def test_corrupt_header_is_rejected():
    w = synth.normal(5000, seed=2)
    c = _encoded(w)
    for off in (0, 4, 8, 24, 28, 56, 88, 96):
        bad = c.copy()
        bad[off] ^= 0x01
        assert oracle.decode(bad)[1] != oracle.OK
    bad = c.copy()
    bad[200] = 1  # reserved bytes must be zero
    assert oracle.decode(bad)[1] == oracle.E_FORMAT
    bad = c.copy()
    s = int(np.argmax(c[256:512]))
    bad[256 + s] += 1  # breaks the Kraft equality
    assert oracle.decode(bad)[1] == oracle.E_FORMAT
    assert oracle.decode(c[:-256])[1] == oracle.E_FORMAT


def test_corrupt_index_is_rejected():
    w = synth.normal(5000, seed=2)
    c = _encoded(w)
    off_chunk = _field(c, "off_chunk")
    off_block = _field(c, "off_block")
    for k in (0, 3, 10):
        for bit in (0, 6):
            bad = c.copy()
            bad[off_chunk + 2 * k] ^= 1 << bit
            assert oracle.decode(bad)[1] == oracle.E_INDEX
    bad = c.copy()
    bad[off_block + 8] ^= 1
    assert oracle.decode(bad)[1] == oracle.E_INDEX


def test_corrupt_stream_is_detected():
    w = synth.normal(5000, seed=2)
    c = _encoded(w)
    off_exp = _field(c, "off_exp")
    for byte in (0, 17, 100, 301):
        bad = c.copy()
        bad[off_exp + byte] ^= 0x10
        out, st = oracle.decode(bad)
        assert st != oracle.OK or not np.array_equal(out, w)
