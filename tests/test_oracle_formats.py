"""Pins for the oracle's other element formats: FP16 and E4M3 in the same
container as BF16.

The hand-derived golden containers fix each format's split into a coded
symbol and raw bits, the nibble order of the E4M3 raw section and the
format field of the header.  The value-based checks fix the split against
the numbers the bits stand for (numpy's float16 for FP16; the E4M3
definition -- bias 7, 3 mantissa bits, largest value 448 -- through the
generator's value-to-bits rounding), so a field taken from the wrong bits
fails.  Exhaustive and brute-force round trips fix losslessness over every
bit pattern of both formats.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from weight_streaming_canonical_gb300 import synth

FP16, E4M3 = oracle.FMT_FP16, oracle.FMT_E4M3


def _le(c, off, nb):
    return int.from_bytes(c[off:off + nb].tobytes(), "little")


HEADER_FIELDS = {
    "n": (8, 8), "total_bits": (16, 8), "T": (24, 4), "C": (28, 4), "n_chunks": (32, 8),
    "n_blocks": (40, 8), "off_exp": (48, 8), "exp_bytes": (56, 8), "off_sm": (64, 8),
    "off_chunk": (72, 8), "off_block": (80, 8), "container_bytes": (88, 8), "longest": (96, 4),
    "nsym": (100, 4), "fill": (104, 4), "format": (108, 4), "off_hi": (112, 8),
}


def _lengths(d):
    lens = np.zeros(256, np.uint8)
    for k, v in d.items():
        lens[int(k)] = v
    return lens


@pytest.mark.parametrize("name,dtype", [("container_fp16_tiny.json", np.uint16), ("container_e4m3_tiny.json", np.uint8)])
def test_golden_format_containers(golden_dir, name, dtype):
    g = json.load(open(os.path.join(golden_dir, name)))
    fmt = g["format"]
    w = np.array([int(h, 16) for h in g["elements_hex"]], dtype)
    h = oracle.histogram(w, fmt)
    expect = np.bincount(np.array(g["symbols"]), minlength=256)
    assert np.array_equal(h, expect)
    c = oracle.encode(w, _lengths(g["lengths"]), g["T"], g["C"], fmt=fmt)
    assert c.size == g["header"]["container_bytes"]
    for k, v in g["header"].items():
        off, nb = HEADER_FIELDS[k]
        assert _le(c, off, nb) == v, k
    assert not c[120:256].any()
    assert _le(c, 112, 8) == g["header"].get("off_hi", 0)
    off_exp = g["header"]["off_exp"]
    words = [_le(c, off_exp + 4 * i, 4) for i in range(len(g["stream_words_hex"]))]
    assert words == [int(x, 16) for x in g["stream_words_hex"]]
    raw = c[g["header"]["off_sm"]: g["header"]["off_sm"] + len(g["raw_hex"])]
    assert raw.tolist() == [int(x, 16) for x in g["raw_hex"]]
    raw_end = g["header"].get("off_hi") or g["header"]["off_chunk"]
    assert not c[g["header"]["off_sm"] + len(g["raw_hex"]): raw_end].any()
    if "hi_hex" in g:
        off_hi = g["header"]["off_hi"]
        hi = c[off_hi: off_hi + len(g["hi_hex"])]
        assert hi.tolist() == [int(x, 16) for x in g["hi_hex"]]
        assert not c[off_hi + len(g["hi_hex"]): g["header"]["off_chunk"]].any()
    entries = [_le(c, g["header"]["off_chunk"] + 2 * i, 2) for i in range(g["header"]["n_chunks"])]
    assert entries == g["chunk_entries"]
    blocks = [_le(c, g["header"]["off_block"] + 8 * i, 8) for i in range(g["header"]["n_blocks"] + 1)]
    assert blocks == g["block_index"]
    out, st = oracle.decode(c)
    assert st == oracle.OK and out.dtype == dtype and out.tolist() == w.tolist()


# ---- FP16: the fields from the value ------------------------------------------------

def _fp16_fields(bits):
    """(biased exponent, 10-bit fraction, sign) of float16 values, from the numbers themselves."""
    x = bits.view(np.float16).astype(np.float64)
    a = np.abs(x)
    exp = np.zeros(a.size, np.int64)
    frac = np.zeros(a.size, np.int64)
    normal = a >= 2.0 ** -14
    m, ex = np.frexp(a[normal])          # a = m 2^ex, m in [0.5, 1)
    k = ex - 1                           # floor(log2 a)
    exp[normal] = k + 15
    frac[normal] = np.rint((a[normal] / np.ldexp(1.0, k) - 1.0) * 1024).astype(np.int64)
    sub = ~normal                        # exponent field 0: a = fraction * 2^-24
    frac[sub] = np.rint(a[sub] / 2.0 ** -24).astype(np.int64)
    return exp, frac, np.signbit(x).astype(np.int64), normal


def test_fp16_symbol_is_the_exponent_by_value():
    bits = synth.normal_fp16(200_000, 0.0, 0.02, seed=3)
    bits = np.concatenate([bits, synth.normal_fp16(50_000, 0.0, 3e-5, seed=4)])  # many subnormals
    finite = np.isfinite(bits.view(np.float16))
    bits = bits[finite]
    exp, _, _, normal = _fp16_fields(bits)
    assert (~normal).sum() > 1000
    assert np.array_equal(oracle.histogram(bits, FP16), np.bincount(exp, minlength=256))


def test_fp16_raw_byte_and_hi_section_by_value():
    bits = synth.normal_fp16(4097, 0.0, 0.5, seed=5)
    exp, frac, sign, _ = _fp16_fields(bits)
    lens = oracle.code_lengths(oracle.histogram(bits, FP16))
    c = oracle.encode(bits, lens, fmt=FP16)
    off_sm, off_hi, off_chunk = _le(c, 64, 8), _le(c, 112, 8), _le(c, 72, 8)
    assert off_hi >= off_sm + bits.size and off_chunk >= off_hi + (bits.size + 1) // 2
    # sign and the 7 trailing fraction bits, one byte per element
    assert c[off_sm: off_sm + bits.size].tolist() == ((sign << 7) | (frac & 0x7F)).tolist()
    # the 3 leading fraction bits: element i in nibble i (low nibble first), bit 3 zero
    sec = c[off_hi: off_hi + (bits.size + 1) // 2]
    nib = np.stack([sec & 0xF, sec >> 4], axis=1).reshape(-1)
    assert nib[: bits.size].astype(np.int64).tolist() == (frac >> 7).tolist()
    assert not nib[bits.size:].any()


@pytest.mark.parametrize("T", [4, 32])
def test_fp16_exhaustive_all_patterns(T):
    w = synth.all_bf16_patterns()  # every 16-bit pattern, read as FP16
    lens = oracle.code_lengths(oracle.histogram(w, FP16))
    c = oracle.encode(w, lens, T, 32 if T == 4 else 256, fmt=FP16)
    out, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(out, w)
    assert oracle.header_format(c) == FP16


# ---- E4M3: the symbol and the nibble from the value ------------------------------------

def _e4m3_values():
    """Every finite E4M3 value as a number: +-(1 + m/8) 2^k, k = -6..8 (448 the
    largest), and the subnormals +-m 2^-9."""
    vals, exps, mants = [], [], []
    for k in range(-6, 9):
        for m in range(8):
            if k == 8 and m == 7:
                continue  # that pattern is NaN
            vals.append((1 + m / 8) * 2.0 ** k)
            exps.append(k + 7)
            mants.append(m)
    for m in range(8):
        vals.append(m * 2.0 ** -9)
        exps.append(0)
        mants.append(m)
    return np.array(vals), np.array(exps), np.array(mants)


def test_e4m3_known_encodings():
    # values fixed by the E4M3 definition: bias 7, 3 mantissa bits, largest 448
    v = np.array([1.0, 2.0, 0.5, 448.0, 2.0 ** -6, 2.0 ** -9, -1.0, 0.0, 240.0], np.float32)
    assert synth.e4m3_round(v).tolist() == [0x38, 0x40, 0x30, 0x7E, 0x08, 0x01, 0xB8, 0x00, 0x77]


def test_e4m3_symbol_and_nibble_by_value():
    vals, exps, mants = _e4m3_values()
    rng = np.random.default_rng(6)
    sign = rng.integers(0, 2, vals.size)
    signed = np.where(sign == 1, -vals, vals)
    bits = synth.e4m3_round(signed.astype(np.float32))
    # exact values come out of the rounding as the definition's fields
    assert ((bits & 0x7F).astype(np.int64) == ((exps << 3) | mants)).all()
    assert np.array_equal(oracle.histogram(bits, E4M3), np.bincount(exps, minlength=256))
    lens = oracle.code_lengths(oracle.histogram(bits, E4M3))
    c = oracle.encode(bits, lens, fmt=E4M3)
    off_sm = _le(c, 64, 8)
    raw = c[off_sm: off_sm + (bits.size + 1) // 2]
    nib = np.empty(raw.size * 2, np.int64)
    nib[0::2] = raw & 0xF   # element 2k in the low nibble of byte k
    nib[1::2] = raw >> 4
    # a zero of either sign carries its sign bit like any other value
    expect = (sign.astype(np.int64) << 3) | mants
    assert nib[: bits.size].tolist() == expect.tolist()
    out, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(out, bits)


@pytest.mark.parametrize("n", [1, 2, 3, 255, 256, 257, 4097])
def test_e4m3_all_patterns_ragged(n):
    rng = np.random.default_rng(n)
    w = np.resize(rng.permutation(synth.all_e4m3_patterns()), n)
    lens = oracle.code_lengths(oracle.histogram(w, E4M3))
    c = oracle.encode(w, lens, 4, 32, fmt=E4M3)
    out, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(out, w)
    assert _le(c, 72, 8) - _le(c, 64, 8) >= (n + 1) // 2  # raw section: one nibble per element


def test_e4m3_brute_force_tiny_tensors():
    alphabet = np.array([0x00, 0x38, 0xC1, 0x7F, 0x01], np.uint8)  # zero, 1.0, -2.25, NaN, smallest subnormal
    for k in range(1, 4):
        for combo in itertools.product(range(alphabet.size), repeat=k):
            w = alphabet[list(combo)]
            lens = oracle.code_lengths(oracle.histogram(w, E4M3))
            c = oracle.encode(w, lens, 4, 32, fmt=E4M3)
            out, st = oracle.decode(c)
            assert st == oracle.OK and np.array_equal(out, w), combo


def test_e4m3_single_binade_needs_no_stream():
    # every element in [1, 2): one exponent, no code bits; the raw section is ceil(n / 2) bytes
    w = synth.e4m3_round(np.linspace(1.0, 1.875, 8, dtype=np.float32))
    w = np.resize(w, 1001)
    lens = oracle.code_lengths(oracle.histogram(w, E4M3))
    assert lens.max() == 0
    c = oracle.encode(w, lens, fmt=E4M3)
    assert _le(c, 16, 8) == 0 and _le(c, 100, 4) == 1 and _le(c, 104, 4) == 7
    out, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(out, w)


@pytest.mark.parametrize("fmt,gen", [(FP16, lambda: synth.normal_fp16(1 << 18, seed=7)),
                                     (E4M3, lambda: synth.normal_e4m3(1 << 18, seed=7))])
def test_entropy_bound(fmt, gen):
    w = gen()
    h = oracle.histogram(w, fmt).astype(np.float64)
    lens = oracle.code_lengths(h.astype(np.uint64))
    p = h[h > 0] / h.sum()
    H = -(p * np.log2(p)).sum()
    L = (h * lens).sum() / h.sum()
    assert H <= L < H + 1
    assert L <= H * 1.01 + 0.02  # near the entropy for these smooth distributions


# ---- rejects ------------------------------------------------------------------------

def _tiny_e4m3():
    w = np.array([0x38, 0xC1, 0x3C, 0x30, 0x3E], np.uint8)
    lens = oracle.code_lengths(oracle.histogram(w, E4M3))
    return w, lens, oracle.encode(w, lens, 4, 32, fmt=E4M3)


def test_e4m3_rejects_a_length_past_the_symbol_range():
    w, lens, c = _tiny_e4m3()
    bad = lens.copy()
    bad[16] = 3
    with pytest.raises(ValueError):
        oracle.encode(w, bad, 4, 32, fmt=E4M3)
    c2 = c.copy()
    c2[256 + 16] = 3
    assert oracle.decode(c2)[1] == oracle.E_FORMAT


def test_e4m3_rejects_a_used_padding_nibble():
    w, lens, c = _tiny_e4m3()
    c2 = c.copy()
    c2[_le(c, 64, 8) + 2] |= 0x50
    assert oracle.decode(c2)[1] == oracle.E_FORMAT


def test_unknown_format_is_rejected():
    w, lens, c = _tiny_e4m3()
    c2 = c.copy()
    c2[108] = 3
    assert oracle.decode(c2)[1] == oracle.E_FORMAT
    with pytest.raises(ValueError):
        oracle.encode(w.astype(np.uint16), lens, fmt=3)


def test_e4m3_single_symbol_fill_in_range():
    w = np.full(9, 0x38, np.uint8)
    lens = np.zeros(256, np.uint8)
    c = oracle.encode(w, lens, fmt=E4M3)
    assert _le(c, 104, 4) == 7
    c2 = c.copy()
    c2[104] = 16
    assert oracle.decode(c2)[1] == oracle.E_FORMAT


def test_fp16_rejects_a_used_hi_padding_bit():
    w = np.array([0x3C00, 0xBE00, 0x3780, 0x3C01, 0x4000], np.uint16)  # 5 hi nibbles in 3 bytes
    lens = oracle.code_lengths(oracle.histogram(w, FP16))
    c = oracle.encode(w, lens, 4, 32, fmt=FP16)
    assert oracle.decode(c)[1] == oracle.OK
    c2 = c.copy()
    c2[_le(c, 112, 8) + 2] |= 0x10  # the nibble past element 4
    assert oracle.decode(c2)[1] == oracle.E_FORMAT
    for byte, bit in ((0, 0x08), (0, 0x80), (2, 0x08)):  # bit 3 of element 0's, 1's and 4's nibble
        c4 = c.copy()
        c4[_le(c, 112, 8) + byte] |= bit
        assert oracle.decode(c4)[1] == oracle.E_FORMAT
    c3 = c.copy()
    c3[112] ^= 0x01  # the hi section's offset no longer matches the layout
    assert oracle.decode(c3)[1] == oracle.E_FORMAT
