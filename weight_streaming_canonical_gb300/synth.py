"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws random BF16 bit patterns (and FP16 or E4M3 ones for the
other element formats) with the shapes and value distributions of the
workloads.  It holds none of the codec's arithmetic:
no exponent split, no code construction, no packing.

Shapes follow "Memory requirements of language model inference on a
consumer GPU": Table 2 (vocabulary 151,936, hidden size 5,120, 40 decoder
layers, 8 key/value heads of 128) and Table 4 (about 330M weights per
decoder layer, 778M each for the embedding table and the output head,
14.8B / 29.5 GB in total).  The feed-forward width 17,408 is not on that
page; it is the Qwen3-14B value this library's workloads use.  Real
checkpoint weights are not used: every value is drawn from a seeded
distribution (normal with std 0.02 for matrices, mean 1 / std 0.05 for the
two norm vectors, a heavy-tailed mix for the adversarial tensor).

Every tensor is generated in fixed blocks of 2**24 elements, each block from
its own seeded PCG64 stream, so any tensor (or block) can be regenerated on
its own and blocks can be drawn in parallel threads.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

BLOCK = 1 << 24

VOCAB = 151_936
HIDDEN = 5_120
LAYERS = 40
KV_HEADS = 8
HEAD_DIM = 128
FFN = 17_408
KV_DIM = KV_HEADS * HEAD_DIM  # 1024

# One decoder layer, in execution order.  Shape is [out][in] (a row of a
# matrix is one output, PyTorch nn.Linear layout); norms are vectors.
LAYER_TENSORS = (
    ("input_layernorm", (HIDDEN,), "norm"),
    ("q_proj", (HIDDEN, HIDDEN), "matrix"),
    ("k_proj", (KV_DIM, HIDDEN), "matrix"),
    ("v_proj", (KV_DIM, HIDDEN), "matrix"),
    ("o_proj", (HIDDEN, HIDDEN), "matrix"),
    ("post_attention_layernorm", (HIDDEN,), "norm"),
    ("gate_proj", (FFN, HIDDEN), "matrix"),
    ("up_proj", (FFN, HIDDEN), "matrix"),
    ("down_proj", (HIDDEN, FFN), "matrix"),
)
EMBED_SHAPE = (VOCAB, HIDDEN)
HEAD_SHAPE = (VOCAB, HIDDEN)

# stream ids keep the tensors of one seed independent of one another
_TENSOR_IDS = {name: i for i, (name, _, _) in enumerate(LAYER_TENSORS)}
_EMBED_ID, _HEAD_ID, _MATRIX_ID, _ADVERSARIAL_ID, _ACT_ID = 100, 101, 102, 103, 104


def numel(shape) -> int:
    out = 1
    for s in shape:
        out *= int(s)
    return out


def layer_weight_count() -> int:
    return sum(numel(shape) for _, shape, _ in LAYER_TENSORS)


def model_weight_count() -> int:
    return LAYERS * layer_weight_count() + numel(EMBED_SHAPE) + numel(HEAD_SHAPE)


def bf16_round(f: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns (uint16), round to nearest even; NaN stays NaN."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    u = f.view(np.uint32)
    r = u >> np.uint32(16)
    r &= np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    out = r.astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = ((u[nan] >> np.uint32(16)) | np.uint32(0x40)).astype(np.uint16)
    return out


def _rng(seed: int, stream: int, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream), int(block)])))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def fp16_round(f: np.ndarray) -> np.ndarray:
    """float32 -> IEEE binary16 bit patterns (uint16), round to nearest even
    (numpy's conversion); magnitudes past 65504 become infinities."""
    with np.errstate(over="ignore"):
        return np.ascontiguousarray(f, dtype=np.float32).astype(np.float16).view(np.uint16)


E4M3_MAX = 448.0  # largest finite OCP E4M3 value, 1.75 * 2**8


def e4m3_round(f: np.ndarray) -> np.ndarray:
    """float32 -> OCP 8-bit float E4M3 bit patterns (uint8): 1 sign, 4 exponent
    bits with bias 7, 3 mantissa bits; round to nearest even, magnitudes past
    448 saturate to 448 (the format has no infinities).  NaN is not produced."""
    x = np.ascontiguousarray(f, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
    a = np.minimum(np.abs(x), E4M3_MAX)
    out = np.zeros(a.shape, np.uint8)
    normal = a >= 2.0 ** -6
    # subnormals: multiples of 2**-9 below 2**-6 (a result of 8 is the smallest normal)
    q = np.rint(a[~normal] / 2.0 ** -9).astype(np.int64)
    out[~normal] = np.where(q >= 8, np.uint8(1 << 3), q.astype(np.uint8))
    an = a[normal]
    e = np.floor(np.log2(an)).astype(np.int64)
    # log2 of a value just below a power of two can round up: fix the exponent exactly
    e = np.where(np.ldexp(1.0, e) > an, e - 1, e)
    e = np.where(np.ldexp(1.0, e + 1) <= an, e + 1, e)
    m = np.rint((an / np.ldexp(1.0, e) - 1.0) * 8.0).astype(np.int64)
    carry = m == 8
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 0, m)
    big = (e > 8) | ((e == 8) & (m > 6))
    e = np.where(big, 8, e)
    m = np.where(big, 6, m)
    out[normal] = (((e + 7) << 3) | m).astype(np.uint8)
    return out | sign


def _blocked(n: int, fill, seed: int, stream: int, dtype=np.uint16) -> np.ndarray:
    out = np.empty(n, dtype)
    starts = list(range(0, n, BLOCK))

    def work(start: int) -> None:
        stop = min(n, start + BLOCK)
        out[start:stop] = fill(_rng(seed, stream, start // BLOCK), stop - start)

    if len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, starts))
    return out


def normal(n: int, mean: float = 0.0, std: float = 0.02, seed: int = 0, stream: int = _MATRIX_ID) -> np.ndarray:
    """n BF16 patterns of N(mean, std) drawn in float32 and rounded to nearest even."""

    def fill(rng, k):
        v = rng.standard_normal(k, dtype=np.float32)
        v *= np.float32(std)
        v += np.float32(mean)
        return bf16_round(v)

    return _blocked(int(n), fill, seed, stream)


def normal_fp16(n: int, mean: float = 0.0, std: float = 0.02, seed: int = 0, stream: int = _MATRIX_ID) -> np.ndarray:
    """n FP16 patterns of N(mean, std) drawn in float32 and rounded to nearest even."""

    def fill(rng, k):
        v = rng.standard_normal(k, dtype=np.float32)
        v *= np.float32(std)
        v += np.float32(mean)
        return fp16_round(v)

    return _blocked(int(n), fill, seed, stream)


def normal_e4m3(n: int, mean: float = 0.0, std: float = 1.0, seed: int = 0, stream: int = _MATRIX_ID) -> np.ndarray:
    """n E4M3 patterns of N(mean, std) * 448 / (6 std): a per-tensor scale that puts
    six standard deviations at the format's largest value, the usual way FP8
    weights are stored (the scale is kept beside the tensor, not in it)."""
    scale = E4M3_MAX / (6.0 * std)

    def fill(rng, k):
        v = rng.standard_normal(k, dtype=np.float32).astype(np.float64) * std + mean
        return e4m3_round((v * scale).astype(np.float32))

    return _blocked(int(n), fill, seed, stream, np.uint8)


def adversarial(n: int = 1 << 28, seed: int = 0, stream: int = _ADVERSARIAL_ID) -> np.ndarray:
    """Heavy-tailed BF16 tensor with every special pattern class.

    Student-t (3 degrees of freedom) x 0.01; 1 % of elements x 100; 5 %
    exact zeros of random sign; 1e-4 subnormals (random sign, mantissa
    1..127); 1e-5 infinities of random sign; 1e-5 NaNs (random sign,
    payload 1..127, so both quiet and signalling).
    """

    def fill(rng, k):
        v = (rng.standard_t(3.0, size=k) * 0.01).astype(np.float32)
        u = rng.random(k)
        sign = (rng.integers(0, 2, size=k, dtype=np.uint16) << np.uint16(15)).astype(np.uint16)
        payload = rng.integers(1, 128, size=k, dtype=np.uint16)
        outlier = (u >= 0.05 + 1e-4 + 2e-5) & (u < 0.06 + 1e-4 + 2e-5)
        v[outlier] *= np.float32(100.0)
        bits = bf16_round(v)
        zero = u < 0.05
        sub = (u >= 0.05) & (u < 0.05 + 1e-4)
        inf = (u >= 0.05 + 1e-4) & (u < 0.05 + 1e-4 + 1e-5)
        nan = (u >= 0.05 + 1e-4 + 1e-5) & (u < 0.05 + 1e-4 + 2e-5)
        bits[zero] = sign[zero]
        bits[sub] = sign[sub] | payload[sub]
        bits[inf] = sign[inf] | np.uint16(0x7F80)
        bits[nan] = sign[nan] | np.uint16(0x7F80) | payload[nan]
        return bits

    return _blocked(int(n), fill, seed, stream)


def matrix_4096(seed: int = 0) -> np.ndarray:
    """Single 4096 x 4096 BF16 matrix, N(0, 0.02)."""
    return normal(4096 * 4096, 0.0, 0.02, seed, _MATRIX_ID).reshape(4096, 4096)


def layer_tensor(name: str, seed: int = 0, layer: int = 0) -> np.ndarray:
    for nm, shape, kind in LAYER_TENSORS:
        if nm == name:
            stream = 1000 + 16 * int(layer) + _TENSOR_IDS[nm]
            if kind == "norm":
                return normal(numel(shape), 1.0, 0.05, seed, stream).reshape(shape)
            return normal(numel(shape), 0.0, 0.02, seed, stream).reshape(shape)
    raise KeyError(name)


def layer_tensor_fp16(name: str, seed: int = 0, layer: int = 0) -> np.ndarray:
    """The layer tensor `name` with the same value distribution, stored as FP16."""
    for nm, shape, kind in LAYER_TENSORS:
        if nm == name:
            stream = 2000 + 16 * int(layer) + _TENSOR_IDS[nm]
            if kind == "norm":
                return normal_fp16(numel(shape), 1.0, 0.05, seed, stream).reshape(shape)
            return normal_fp16(numel(shape), 0.0, 0.02, seed, stream).reshape(shape)
    raise KeyError(name)


def layer_matrix_e4m3(name: str, seed: int = 0, layer: int = 0) -> np.ndarray:
    """The layer matrix `name` stored as E4M3 with a per-tensor scale (matrices
    only: the norm vectors stay in a wider format)."""
    for nm, shape, kind in LAYER_TENSORS:
        if nm == name:
            if kind != "matrix":
                raise KeyError(f"{name} is not a matrix")
            stream = 3000 + 16 * int(layer) + _TENSOR_IDS[nm]
            return normal_e4m3(numel(shape), 0.0, 0.02, seed, stream).reshape(shape)
    raise KeyError(name)


def layer(seed: int = 0, layer_index: int = 0) -> dict[str, np.ndarray]:
    """All tensors of one Qwen3-14B-shaped decoder layer (~330M weights)."""
    return {name: layer_tensor(name, seed, layer_index) for name, _, _ in LAYER_TENSORS}


def embedding(seed: int = 0) -> np.ndarray:
    return normal(numel(EMBED_SHAPE), 0.0, 0.02, seed, _EMBED_ID).reshape(EMBED_SHAPE)


def lm_head(seed: int = 0) -> np.ndarray:
    return normal(numel(HEAD_SHAPE), 0.0, 0.02, seed, _HEAD_ID).reshape(HEAD_SHAPE)


def activations(batch: int, width: int, seed: int = 1, stream: int = _ACT_ID) -> np.ndarray:
    """[batch][width] BF16 activation vectors, N(0, 1)."""
    return normal(batch * width, 0.0, 1.0, seed, stream).reshape(batch, width)


def exponent_mix(n: int, n_exponents: int, ratio: float = 0.85, first: int = 100, seed: int = 0) -> np.ndarray:
    """n BF16 patterns whose exponents are first .. first + n_exponents - 1,
    exponent first + k drawn with probability proportional to ratio**k;
    sign and mantissa uniform.  Sets the size and shape of the code tree
    directly (every exponent is present once n is large enough)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), 105, int(n_exponents)])))
    p = ratio ** np.arange(n_exponents, dtype=np.float64)
    p /= p.sum()
    e = (first + rng.choice(n_exponents, size=int(n), p=p)).astype(np.uint16)
    low = rng.integers(0, 1 << 16, size=int(n), dtype=np.uint32).astype(np.uint16)
    return (low & np.uint16(0x807F)) | (e << np.uint16(7))


def long_tail(n: int, tail: float = 1e-3, seed: int = 0) -> np.ndarray:
    """N(0, 0.02) BF16 weights with a share `tail` of them (chosen uniformly,
    sign and mantissa kept) given an exponent drawn uniformly from 1..254:
    the shape of a checkpoint with rare outliers across the whole range, a
    code tree of about 250 internal nodes whose deep nodes are rarely
    reached."""
    w = normal(n, seed=seed)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), 107])))
    pick = rng.choice(int(n), size=int(n * tail), replace=False)
    e = rng.integers(1, 255, size=pick.size).astype(np.uint16)
    w[pick] = (w[pick] & np.uint16(0x807F)) | (e << np.uint16(7))
    return w


def all_bf16_patterns() -> np.ndarray:
    """Every one of the 65,536 BF16 bit patterns, in order."""
    return np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def all_e4m3_patterns() -> np.ndarray:
    """Every one of the 256 E4M3 bit patterns, in order (0x7F and 0xFF are NaN)."""
    return np.arange(256, dtype=np.uint16).astype(np.uint8)
