"""Host side of the library (no GPU): the encoder against the oracle, header
validation, geometry choice, and the exported C ABI."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from weight_streaming_canonical_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cost(hist, lens):
    return int(sum(int(hist[s]) * int(lens[s]) for s in range(256)))


def test_every_declared_entry_point_is_exported(afx):
    header = open(os.path.join(ROOT, "include", "afx.h")).read()
    body = re.sub(r"/\*.*?\*/", "", header, flags=re.S)
    names = set(re.findall(r"\b(afx_[a-z_]+)\s*\(", body))
    assert {"afx_build_code", "afx_encode_bound", "afx_encode", "afx_decode", "afx_decode_gemv",
            "afx_stream_run", "afx_parse_header"} <= names
    lib = ctypes.CDLL(afx.LIB_PATH)
    for name in sorted(names):
        assert hasattr(lib, name), name


def test_struct_sizes_match_the_c_layout(afx):
    # afx_code: 256 u64 + 256 u32 + 256 u8 + 4 u32; afx_desc: fixed fields + 256 lengths
    assert ctypes.sizeof(afx.afx_code) == 2048 + 1024 + 256 + 16
    assert ctypes.sizeof(afx.afx_desc) == 8 * 2 + 4 * 2 + 8 * 2 + 8 * 7 + 4 * 4 + 256


CASES = {
    "normal": lambda: synth.normal(300_001, seed=1),
    "norm_vector": lambda: synth.normal(5120, 1.0, 0.05, seed=2),
    "all_patterns": synth.all_bf16_patterns,
    "adversarial": lambda: synth.adversarial(1 << 20, seed=3),
    "two_symbols": lambda: np.array([0x3F80, 0x4000] * 999, np.uint16),
    "single": lambda: np.full(777, 0x3F80, np.uint16),
    "empty": lambda: np.zeros(0, np.uint16),
    "tiny": lambda: np.array([0x3F80, 0x0001, 0xFFC1], np.uint16),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_code_is_optimal_and_canonical(afx, case):
    w = CASES[case]()
    code = afx.afx_build_code(w)
    hist = oracle.histogram(w)
    assert np.array_equal(np.array(code.count[:], np.uint64), hist)
    lens = np.array(code.len[:], np.uint8)
    ref = oracle.code_lengths(hist, 24)
    assert _cost(hist, lens) == _cost(hist, ref)
    assert lens.max() <= 24
    if code.nsym >= 2:
        assert sum(1 << (24 - int(l)) for l in lens if l) == 1 << 24
    assert np.array_equal(np.array(code.code[:], np.uint32), oracle.canonical_codes(lens))


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("T", [0, 4, 16, 64])
def test_container_is_byte_identical_to_the_oracle(afx, case, T):
    w = CASES[case]()
    code = afx.afx_build_code(w)
    try:
        desc = afx.afx_encode_bound(w.size, code, T, 256)
    except afx.AfxError:
        assert T == 64  # a 64-byte chunk can exceed the block capacity
        return
    c = afx.afx_encode(w, code, desc)
    ref = oracle.encode(w, np.array(code.len[:], np.uint8), desc.chunk_bytes, 256)
    assert np.array_equal(c, ref)
    out, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(out, w)


def test_geometry_choice_respects_block_capacity(afx):
    w = synth.normal(100_000, seed=4)
    d = afx.afx_encode_bound(w.size, afx.afx_build_code(w))
    # shortest code 2 bits: 512 chunks of 16 bytes hold at most 32768 codewords
    assert d.chunk_bytes == 16 and d.block_chunks == 512
    # a dominant exponent gets a 1-bit code: the chunks shrink to 8 bytes
    v = np.where(np.arange(50_000) % 3 == 0, 0x4000, 0x3F80).astype(np.uint16)
    code = afx.afx_build_code(v)
    assert min(l for l in code.len if l) == 1
    d = afx.afx_encode_bound(v.size, code)
    assert d.chunk_bytes == 8
    with pytest.raises(afx.AfxError):
        afx.afx_encode_bound(v.size, code, 16, 512)
    d = afx.afx_encode_bound(w.size, afx.afx_build_code(w), 0, 256)
    assert d.chunk_bytes == 32 and d.block_chunks == 256


def test_parse_header_roundtrip_and_rejections(afx):
    w = synth.normal(70_000, seed=5)
    c, d = afx.encode(w)
    p = afx.afx_parse_header(c)
    assert afx.desc_dict(p) == afx.desc_dict(d)
    # n and total_bits (offsets 8, 16) can change without moving any section;
    # the header alone cannot show that, the kernels check n against the block index
    for off in (0, 4, 6, 24, 28, 32, 40, 56, 64, 88, 96, 100, 104, 150):
        bad = c.copy()
        bad[off] ^= 0x04
        with pytest.raises(afx.AfxError):
            afx.afx_parse_header(bad)
    bad = c.copy()
    bad[256 + int(np.argmax(c[256:512]))] += 1  # Kraft equality broken
    with pytest.raises(afx.AfxError):
        afx.afx_parse_header(bad)
    with pytest.raises(afx.AfxError):
        afx.afx_parse_header(c[:100])


def test_encode_rejects_data_the_code_does_not_cover(afx):
    w = synth.normal(10_000, seed=6)
    code = afx.afx_build_code(w)
    desc = afx.afx_encode_bound(w.size, code)
    other = w.copy()
    other[17] = 0x7F80  # +inf: exponent 255, absent from the code
    with pytest.raises(afx.AfxError):
        afx.afx_encode(other, code, desc)
    with pytest.raises(afx.AfxError):
        afx.afx_encode(w, code, desc, out=np.zeros(desc.container_bytes - 256, np.uint8))


def test_gemv_workspace_size(afx):
    w = synth.normal(5120 * 64, seed=7)
    _, d = afx.encode(w)
    for b in (1, 2, 3, 4):
        assert afx.afx_decode_gemv_workspace(d, b) >= d.n_blocks * 2 * b * 4
    with pytest.raises(afx.AfxError):
        afx.afx_decode_gemv_workspace(d, 5)


# ---- other element formats -------------------------------------------------------

FMT_CASES = {
    "fp16_normal": (1, lambda: synth.normal_fp16(300_001, seed=11)),
    "fp16_all_patterns": (1, synth.all_bf16_patterns),
    "fp16_norm_vector": (1, lambda: synth.normal_fp16(5120, 1.0, 0.05, seed=12)),
    "fp16_single": (1, lambda: np.full(333, 0x3C00, np.uint16)),
    "e4m3_normal": (2, lambda: synth.normal_e4m3(300_001, seed=13)),
    "e4m3_all_patterns": (2, lambda: np.resize(synth.all_e4m3_patterns(), 1027)),
    "e4m3_single": (2, lambda: np.resize(np.array([0x38, 0xB9, 0x3F], np.uint8), 501)),
    "e4m3_tiny_odd": (2, lambda: np.array([0x38, 0xC1, 0x3C, 0x30, 0x3E], np.uint8)),
    "e4m3_empty": (2, lambda: np.zeros(0, np.uint8)),
}


@pytest.mark.parametrize("case", sorted(FMT_CASES))
@pytest.mark.parametrize("T", [0, 4, 16])
def test_format_container_is_byte_identical_to_the_oracle(afx, case, T):
    fmt, gen = FMT_CASES[case]
    w = gen()
    code = afx.afx_build_code_fmt(w, fmt)
    assert code.format == fmt
    hist = oracle.histogram(w, fmt)
    assert np.array_equal(np.array(code.count[:], np.uint64), hist)
    lens = np.array(code.len[:], np.uint8)
    assert _cost(hist, lens) == _cost(hist, oracle.code_lengths(hist, 24))
    desc = afx.afx_encode_bound(w.size, code, T, 256)
    assert desc.format == fmt
    c = afx.afx_encode(w, code, desc)
    ref = oracle.encode(w, lens, desc.chunk_bytes, 256, fmt=fmt)
    assert np.array_equal(c, ref)
    out, st = oracle.decode(c)
    assert st == oracle.OK and np.array_equal(out, w)
    assert afx.desc_dict(afx.afx_parse_header(c)) == afx.desc_dict(desc)


def test_format_rejections(afx):
    w = synth.normal_e4m3(10_000, seed=14)
    c, d = afx.encode(w, fmt=afx.AFX_FMT_E4M3)
    # a code length for a symbol E4M3 cannot produce, an out-of-range fill, an unknown format
    for off, val in ((256 + 16, 3), (108, 3)):
        bad = c.copy()
        bad[off] = val
        with pytest.raises(afx.AfxError):
            afx.afx_parse_header(bad)
    one = np.full(64, 0x38, np.uint8)
    c1, d1 = afx.encode(one, fmt=afx.AFX_FMT_E4M3)
    assert d1.nsym == 1 and d1.fill == 7
    bad = c1.copy()
    bad[104] = 16
    with pytest.raises(afx.AfxError):
        afx.afx_parse_header(bad)
    # the code and the plan must agree on the format
    code16 = afx.afx_build_code_fmt(synth.normal_fp16(1000, seed=1), afx.AFX_FMT_FP16)
    desc16 = afx.afx_encode_bound(1000, code16)
    desc16.format = afx.AFX_FMT_BF16
    with pytest.raises(afx.AfxError):
        afx.afx_encode(synth.normal_fp16(1000, seed=1), code16, desc16)
    with pytest.raises(afx.AfxError):
        afx.afx_build_code_fmt(np.zeros(4, np.uint16), 7)
    # an E4M3 container's raw section is one nibble per element
    assert d.off_chunk - d.off_sm >= (w.size + 1) // 2 and d.off_chunk - d.off_sm < (w.size + 1) // 2 + 256


def test_bf16_containers_are_unchanged_by_the_format_field(afx):
    # format 0 leaves header byte 108 zero: a BF16 container is the same bytes as before the field
    w = synth.normal(20_000, seed=15)
    c, d = afx.encode(w)
    assert d.format == afx.AFX_FMT_BF16 and not c[108:112].any()
    c2, d2 = afx.encode(w, fmt=afx.AFX_FMT_BF16)
    assert np.array_equal(c, c2)


def test_container_survives_a_file_round_trip(afx, tmp_path):
    # the container is the persistence format: bytes written to a file and
    # read back parse to the same description and decode to the same weights
    w = synth.normal(123_457, seed=19)
    c, d = afx.encode(w)
    path = tmp_path / "tensor.afx"
    c.tofile(path)
    back = np.fromfile(path, dtype=np.uint8)
    assert np.array_equal(back, c)
    assert afx.desc_dict(afx.afx_parse_header(back)) == afx.desc_dict(d)
    out, st = oracle.decode(back)
    assert st == oracle.OK and np.array_equal(out, w)


@pytest.mark.parametrize("fmt,n,T", [(0, 6_000_011, 0), (0, 5_000_000, 4), (1, 4_000_003, 16), (2, 3_000_017, 8),
                                     (0, 2_097_152, 4)])
def test_parallel_encoder_is_byte_identical_to_the_oracle(afx, fmt, n, T):
    # large enough for several encoder threads (one per million elements):
    # the segment edges, shared stream words and shared chunk entries merge
    # to the oracle's single-pass container
    w = (synth.normal(n, seed=n) if fmt == 0 else synth.normal_fp16(n, seed=n) if fmt == 1
         else synth.normal_e4m3(n, seed=n))
    code = afx.afx_build_code_fmt(w, fmt)
    desc = afx.afx_encode_bound(w.size, code, T, 256 if T == 4 else 0)
    c = afx.afx_encode(w, code, desc)
    ref = oracle.encode(w, np.array(code.len[:], np.uint8), desc.chunk_bytes, desc.block_chunks, fmt=fmt)
    assert np.array_equal(c, ref)


def test_encode_refuses_elements_that_do_not_match_the_plan(afx):
    # the code and plan of one tensor, the elements of another whose codes
    # are longer: refused before any stream byte is written
    w1 = synth.normal(2_000_000, seed=1)
    code = afx.afx_build_code(w1)
    desc = afx.afx_encode_bound(w1.size, code)
    w2 = synth.normal(2_000_000, 0.0, 0.0002, seed=2)  # exponents from the code's rare, long end
    lens = np.array(code.len[:], np.uint8)
    w2 = np.where(lens[(w2 >> 7) & 0xFF] > 0, w2, w1).astype(np.uint16)  # keep every symbol coded
    assert int(lens[(w2 >> 7) & 0xFF].astype(np.int64).sum()) > desc.total_bits
    out = np.zeros(desc.container_bytes, np.uint8)
    with pytest.raises(afx.AfxError):
        afx.afx_encode(w2, code, desc, out=out)
    assert not out[desc.off_exp: desc.off_sm].any()  # nothing of the stream was written
