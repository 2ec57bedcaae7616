"""Pins for the oracle's code construction (package-merge + canonical codes).

Each check comes from outside the oracle: a textbook worked example, brute
force over every admissible length vector, an independent dynamic program
for length-limited codes, Huffman's own heap construction, the Kraft
equality, Shannon's bounds and the prefix property.
"""
import heapq
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle


def _hist(counts: dict) -> np.ndarray:
    h = np.zeros(256, np.uint64)
    for s, c in counts.items():
        h[s] = c
    return h


def _cost(h, lens) -> int:
    return int(sum(int(h[s]) * int(lens[s]) for s in range(256)))


def _heap_huffman_cost(counts) -> int:
    """Huffman 1952: repeatedly merge the two smallest weights; the cost is
    the sum of all merged weights."""
    heap = list(counts)
    heapq.heapify(heap)
    total = 0
    while len(heap) > 1:
        a = heapq.heappop(heap)
        b = heapq.heappop(heap)
        total += a + b
        heapq.heappush(heap, a + b)
    return total


def _heap_huffman_depth(counts) -> int:
    heap = [(c, 0, i) for i, c in enumerate(counts)]
    heapq.heapify(heap)
    nxt = len(counts)
    while len(heap) > 1:
        a = heapq.heappop(heap)
        b = heapq.heappop(heap)
        heapq.heappush(heap, (a[0] + b[0], max(a[1], b[1]) + 1, nxt))
        nxt += 1
    return heap[0][1]


def _brute_force_min_cost(counts, max_len) -> int:
    best = None
    for lens in itertools.product(range(1, max_len + 1), repeat=len(counts)):
        if sum(2.0 ** -l for l in lens) <= 1.0 + 1e-12:
            c = sum(a * b for a, b in zip(counts, lens))
            best = c if best is None or c < best else best
    return best


def _dp_min_cost(counts, max_len) -> int:
    """Optimal length-limited prefix code by dynamic programming.

    Sort weights descending; an optimal code then has non-decreasing
    lengths.  State: (symbols placed, Kraft units used out of 2**max_len,
    last length).  Independent of package-merge."""
    w = sorted(counts, reverse=True)
    m = len(w)
    U = 1 << max_len
    INF = float("inf")
    # f[u][l] = min cost having placed i symbols using u units, last length l
    f = {(0, 1): 0}
    for i in range(m):
        g = {}
        for (u, lo), c in f.items():
            for l in range(lo, max_len + 1):
                uu = u + (1 << (max_len - l))
                if uu > U:
                    continue
                key = (uu, l)
                v = c + w[i] * l
                if v < g.get(key, INF):
                    g[key] = v
        f = g
    return min(f.values())


def _kraft_units(lens, cap=24) -> int:
    return sum(1 << (cap - int(l)) for l in lens if l > 0)


def test_textbook_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "huffman_textbook.json")))
    h = _hist(dict(zip(g["symbols"], g["counts"])))
    lens = oracle.code_lengths(h, 24)
    assert [int(lens[s]) for s in g["symbols"]] == g["lengths"]
    codes = oracle.canonical_codes(lens)
    got = [format(int(codes[s]), "b").zfill(int(lens[s])) for s in g["symbols"]]
    assert got == g["codes_binary"]
    assert _cost(h, lens) == g["expected_bits"]


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_optimality_small_alphabets(seed):
    rng = np.random.default_rng(seed)
    m = int(rng.integers(2, 7))
    max_len = int(rng.integers(max(1, math.ceil(math.log2(m))), 6))
    counts = [int(c) for c in rng.integers(1, 1000, size=m)]
    if seed % 3 == 0:
        counts = [int(c) for c in rng.geometric(0.3, size=m) * rng.integers(1, 50, size=m)]
    syms = rng.choice(256, size=m, replace=False)
    h = _hist(dict(zip(syms.tolist(), counts)))
    lens = oracle.code_lengths(h, max_len)
    assert max(int(l) for l in lens) <= max_len
    assert all(lens[s] > 0 for s in syms)
    assert _kraft_units([lens[s] for s in syms], max_len) == 1 << max_len  # complete code
    assert _cost(h, lens) == _brute_force_min_cost(counts, max_len)


@pytest.mark.parametrize("seed", range(30))
def test_dynamic_program_optimality_when_cap_binds(seed):
    rng = np.random.default_rng(1000 + seed)
    m = int(rng.integers(6, 13))
    # steeply skewed counts make the unconstrained tree deeper than the cap
    counts = [int(2 ** rng.uniform(0, 14)) + 1 for _ in range(m)]
    max_len = max(math.ceil(math.log2(m)), min(6, _heap_huffman_depth(counts) - 1))
    syms = rng.choice(256, size=m, replace=False)
    h = _hist(dict(zip(syms.tolist(), counts)))
    lens = oracle.code_lengths(h, max_len)
    assert max(int(l) for l in lens) <= max_len
    assert _kraft_units([lens[s] for s in syms], max_len) == 1 << max_len
    assert _cost(h, lens) == _dp_min_cost(counts, max_len)


@pytest.mark.parametrize("seed", range(20))
def test_uncapped_equals_heap_huffman(seed):
    rng = np.random.default_rng(2000 + seed)
    m = int(rng.integers(2, 257))
    counts = rng.integers(1, 10 ** 6, size=m)
    counts = [int(c) for c in counts]
    assert _heap_huffman_depth(counts) <= 24
    syms = rng.choice(256, size=m, replace=False)
    h = _hist(dict(zip(syms.tolist(), counts)))
    lens = oracle.code_lengths(h, 24)
    assert _cost(h, lens) == _heap_huffman_cost(counts)


def test_fibonacci_counts_hit_the_24_bit_cap():
    # Fibonacci weights give the deepest possible Huffman tree.
    fib = [1, 1]
    while len(fib) < 40:
        fib.append(fib[-1] + fib[-2])
    assert _heap_huffman_depth(fib) == 39
    h = _hist({s: c for s, c in enumerate(fib)})
    lens = oracle.code_lengths(h, 24)
    assert int(lens.max()) == 24
    assert _kraft_units(lens) == 1 << 24
    # capping costs something but stays close to the unconstrained optimum
    assert _heap_huffman_cost(fib) <= _cost(h, lens) <= _heap_huffman_cost(fib) * 1.01


def test_shannon_bounds():
    rng = np.random.default_rng(7)
    for _ in range(20):
        m = int(rng.integers(2, 200))
        counts = rng.integers(1, 10 ** 5, size=m).astype(np.float64)
        h = _hist(dict(zip(range(m), counts.astype(np.int64).tolist())))
        lens = oracle.code_lengths(h, 24)
        p = counts / counts.sum()
        H = float(-(p * np.log2(p)).sum())
        Lbar = _cost(h, lens) / counts.sum()
        assert H - 1e-12 <= Lbar < H + 1


def test_degenerate_alphabets():
    assert oracle.code_lengths(np.zeros(256, np.uint64)).max() == 0
    h = _hist({127: 1000})
    assert oracle.code_lengths(h).max() == 0  # one symbol needs no bits
    h = _hist({3: 1, 250: 10 ** 9})
    lens = oracle.code_lengths(h)
    assert lens[3] == 1 and lens[250] == 1
    full = _hist({s: 1 for s in range(256)})
    lens = oracle.code_lengths(full)
    assert set(lens.tolist()) == {8}
    with pytest.raises(ValueError):
        oracle.code_lengths(full, 7)  # 256 symbols cannot fit in 7 bits


@pytest.mark.parametrize("seed", range(10))
def test_canonical_codes_are_prefix_free_and_ordered(seed):
    rng = np.random.default_rng(3000 + seed)
    m = int(rng.integers(2, 257))
    syms = rng.choice(256, size=m, replace=False)
    counts = (2 ** rng.uniform(0, 20, size=m)).astype(np.int64) + 1
    h = _hist(dict(zip(syms.tolist(), counts.tolist())))
    lens = oracle.code_lengths(h, 24)
    codes = oracle.canonical_codes(lens)
    present = sorted((int(lens[s]), int(s)) for s in syms)
    words = [format(int(codes[s]), "b").zfill(l) for l, s in present]
    # no code is a prefix of another
    for a, b in itertools.combinations(words, 2):
        assert not a.startswith(b) and not b.startswith(a)
    # in (length, value) order, left-aligned codes strictly increase
    aligned = [int(wd, 2) << (24 - len(wd)) for wd in words]
    assert aligned == sorted(aligned) and len(set(aligned)) == len(aligned)
    # complete code: first code is all zeros, last is all ones
    assert set(words[0]) == {"0"}
    assert set(words[-1]) == {"1"}
