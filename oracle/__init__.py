"""CPU oracle for the lossless BF16 weight unpack (test infrastructure only).

BF16, FP16 and E4M3 elements share the container (see the C file's header
for how each format splits into a coded symbol and raw bits).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The product library never imports it.  The
arithmetic lives in ``afx_oracle.c`` (plain C, one bit or one element at a
time); this module only builds that file with gcc and marshals numpy arrays.

Passages followed (see the C file for the full statement):
  * "Why Weight Offloading Slows Inference", section "Lossless compression:
    fewer bytes to read, more work to unpack" -- shorter codes for common
    BF16 exponents (Huffman, that page's reference [2]); the released bits
    are restored before computation.
  * "Memory requirements of language model inference on a consumer GPU",
    section "Number formats for weights" -- BF16 weights stay exact.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "afx_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liborc.so")

OK, E_FORMAT, E_CORRUPT, E_INDEX, E_ARG = 0, 1, 2, 3, 4
# element formats: BF16; IEEE binary16; OCP 8-bit float E4M3
FMT_BF16, FMT_FP16, FMT_E4M3 = 0, 1, 2
STATUS_NAMES = {0: "ok", 1: "format", 2: "corrupt", 3: "index", 4: "arg"}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile afx_oracle.c into oracle/_build/liborc.so with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        u64p = ctypes.POINTER(ctypes.c_uint64)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        c_u64, c_u32 = ctypes.c_uint64, ctypes.c_uint32
        vp = ctypes.c_void_p
        lib.orc_histogram.argtypes = [u16p, c_u64, u64p]
        lib.orc_histogram_fmt.argtypes = [vp, c_u64, ctypes.c_uint, u64p]
        lib.orc_code_lengths.argtypes = [u64p, ctypes.c_uint, u8p]
        lib.orc_canonical_codes.argtypes = [u8p, u32p]
        lib.orc_container_bytes.argtypes = [c_u64, c_u64, c_u32, c_u32, u64p]
        lib.orc_container_bytes_fmt.argtypes = [c_u64, ctypes.c_uint, c_u64, c_u32, c_u32, u64p]
        lib.orc_encode.argtypes = [u16p, c_u64, u8p, c_u32, c_u32, u8p, c_u64]
        lib.orc_encode_fmt.argtypes = [vp, c_u64, ctypes.c_uint, u8p, c_u32, c_u32, u8p, c_u64]
        lib.orc_decode.argtypes = [u8p, c_u64, vp, c_u64]
        lib.orc_gemv.argtypes = [u16p, c_u64, c_u64, u16p, ctypes.c_uint, f32p, f64p]
        for f in (lib.orc_histogram, lib.orc_histogram_fmt, lib.orc_code_lengths, lib.orc_canonical_codes,
                  lib.orc_container_bytes, lib.orc_container_bytes_fmt, lib.orc_encode, lib.orc_encode_fmt,
                  lib.orc_decode, lib.orc_gemv):
            f.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_u16(w) -> np.ndarray:
    a = np.ascontiguousarray(w)
    if a.dtype != np.uint16:
        raise TypeError(f"expected BF16 bit patterns as uint16, got {a.dtype}")
    return a.reshape(-1)


def _as_elems(w, fmt: int) -> np.ndarray:
    """Element bit patterns: uint16 for BF16 and FP16, uint8 for E4M3."""
    if fmt not in (FMT_BF16, FMT_FP16, FMT_E4M3):
        raise ValueError(f"unknown element format {fmt}")
    a = np.ascontiguousarray(w)
    want = np.uint8 if fmt == FMT_E4M3 else np.uint16
    if a.dtype != want:
        raise TypeError(f"expected {np.dtype(want).name} bit patterns for format {fmt}, got {a.dtype}")
    return a.reshape(-1)


def histogram(w, fmt: int = FMT_BF16) -> np.ndarray:
    """256-bin count of the coded symbol (the exponent field for BF16 and E4M3)."""
    w = _as_elems(w, fmt)
    h = np.zeros(256, np.uint64)
    _load().orc_histogram_fmt(w.ctypes.data_as(ctypes.c_void_p), w.size, fmt, _ptr(h, ctypes.c_uint64))
    return h


def code_lengths(hist, max_len: int = 24) -> np.ndarray:
    """Optimal prefix-code lengths of at most max_len bits (package-merge)."""
    h = np.ascontiguousarray(hist, dtype=np.uint64)
    assert h.size == 256
    out = np.zeros(256, np.uint8)
    st = _load().orc_code_lengths(_ptr(h, ctypes.c_uint64), max_len, _ptr(out, ctypes.c_uint8))
    if st != OK:
        raise ValueError(f"orc_code_lengths failed: {STATUS_NAMES.get(st, st)}")
    return out


def canonical_codes(lengths) -> np.ndarray:
    """Canonical code of every exponent value from the 256 code lengths."""
    ln = np.ascontiguousarray(lengths, dtype=np.uint8)
    out = np.zeros(256, np.uint32)
    st = _load().orc_canonical_codes(_ptr(ln, ctypes.c_uint8), _ptr(out, ctypes.c_uint32))
    if st != OK:
        raise ValueError(f"orc_canonical_codes failed: {STATUS_NAMES.get(st, st)}")
    return out


def container_bytes(n: int, total_bits: int, T: int = 32, C: int = 256, fmt: int = FMT_BF16) -> int:
    v = ctypes.c_uint64(0)
    st = _load().orc_container_bytes_fmt(n, fmt, total_bits, T, C, ctypes.byref(v))
    if st != OK:
        raise ValueError(f"bad geometry T={T} C={C} or format {fmt}")
    return int(v.value)


def encode(w, lengths, T: int = 32, C: int = 256, fmt: int = FMT_BF16) -> np.ndarray:
    """Whole container (uint8) for the element patterns w of format fmt with the given lengths."""
    w = _as_elems(w, fmt)
    ln = np.ascontiguousarray(lengths, dtype=np.uint8)
    h = histogram(w, fmt)
    total_bits = int(np.sum(h.astype(object) * ln.astype(object)))
    size = container_bytes(w.size, total_bits, T, C, fmt)
    out = np.zeros(size, np.uint8)
    st = _load().orc_encode_fmt(w.ctypes.data_as(ctypes.c_void_p), w.size, fmt, _ptr(ln, ctypes.c_uint8), T, C,
                                _ptr(out, ctypes.c_uint8), size)
    if st != OK:
        raise ValueError(f"orc_encode failed: {STATUS_NAMES.get(st, st)}")
    return out


def header_n(container) -> int:
    c = np.ascontiguousarray(container, dtype=np.uint8)
    return int(c[8:16].view(np.uint64)[0])


def header_format(container) -> int:
    c = np.ascontiguousarray(container, dtype=np.uint8)
    return int(c[108:112].view(np.uint32)[0])


def decode(container) -> tuple[np.ndarray, int]:
    """Bit-serial decode; returns (element patterns, status) where status 0 = ok.
    The elements are uint16 for BF16 and FP16 containers, uint8 for E4M3."""
    c = np.ascontiguousarray(container, dtype=np.uint8)
    if c.size < 512:
        return np.zeros(0, np.uint16), E_FORMAT
    n = header_n(c)
    out = np.zeros(n, np.uint8 if header_format(c) == FMT_E4M3 else np.uint16)
    st = _load().orc_decode(_ptr(c, ctypes.c_uint8), c.size, out.ctypes.data_as(ctypes.c_void_p), n)
    return out, int(st)


def gemv(W, x) -> tuple[np.ndarray, np.ndarray]:
    """y[b][r] = sum_c W[r][c] x[b][c] (float64 exact products, float64 sums,
    rounded to float32) and A[b][r] = sum_c |W[r][c] x[b][c]|."""
    W = np.ascontiguousarray(W)
    x = np.ascontiguousarray(x)
    assert W.dtype == np.uint16 and x.dtype == np.uint16 and W.ndim == 2
    if x.ndim == 1:
        x = x.reshape(1, -1)
    rows, cols = W.shape
    B = x.shape[0]
    assert x.shape[1] == cols
    y = np.zeros((B, rows), np.float32)
    A = np.zeros((B, rows), np.float64)
    st = _load().orc_gemv(_ptr(W, ctypes.c_uint16), rows, cols, _ptr(x, ctypes.c_uint16), B,
                          _ptr(y, ctypes.c_float), _ptr(A, ctypes.c_double))
    if st != OK:
        raise ValueError("orc_gemv failed")
    return y, A
