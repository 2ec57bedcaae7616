"""Pins for the synthetic inputs: shapes against the pages' tables, BF16
rounding against a library conversion, determinism and the recipe's mix."""
import numpy as np
import torch

from weight_streaming_canonical_gb300 import synth


def test_qwen3_14b_sizes_match_table_4():
    # "Memory requirements of language model inference on a consumer GPU",
    # Table 4: one decoder layer ~330M weights / 0.66 GB; embedding and head
    # ~778M / 1.6 GB each; total 14.8B / 29.5 GB (BF16, 2 bytes a weight).
    layer = synth.layer_weight_count()
    assert layer == 330_311_680
    assert round(layer / 1e6) == 330 and round(2 * layer / 1e9, 2) == 0.66
    emb = synth.numel(synth.EMBED_SHAPE)
    assert round(emb / 1e6) == 778 and round(2 * emb / 1e9, 1) == 1.6
    assert synth.numel(synth.HEAD_SHAPE) == emb
    total = synth.model_weight_count()
    assert total == 14_768_291_840
    assert round(total / 1e9, 1) == 14.8 and round(2 * total / 1e9, 1) == 29.5
    assert round(synth.LAYERS * layer / 1e9, 1) == 13.2


def test_table_2_config_values():
    assert (synth.VOCAB, synth.HIDDEN, synth.LAYERS, synth.KV_HEADS, synth.HEAD_DIM) == (151_936, 5_120, 40, 8, 128)
    assert synth.KV_DIM == 1024


def test_bf16_round_matches_torch_conversion():
    rng = np.random.default_rng(1)
    f = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32) * np.float32(0.02),
        (rng.standard_normal(10_000) * 1e30).astype(np.float32),
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895314e38, -0.0, 1e-40, np.inf, -np.inf], np.float32),
    ])
    ours = synth.bf16_round(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    nan = synth.bf16_round(np.array([np.nan], np.float32))
    assert (nan[0] & 0x7F80) == 0x7F80 and (nan[0] & 0x7F) != 0


def test_generation_is_deterministic_and_streams_differ():
    a = synth.normal(3 * synth.BLOCK // 2, seed=9)
    b = synth.normal(3 * synth.BLOCK // 2, seed=9)
    assert np.array_equal(a, b)
    c = synth.normal(1000, seed=9, stream=5)
    assert not np.array_equal(a[:1000], c)
    q = synth.layer_tensor("q_proj", seed=0, layer=0)
    q1 = synth.layer_tensor("q_proj", seed=0, layer=1)
    assert q.shape == (5120, 5120) and not np.array_equal(q[:4], q1[:4])


def test_value_distributions():
    w = synth.normal(1 << 20, 0.0, 0.02, seed=3)
    f = (w.astype(np.uint32) << 16).view(np.float32)
    assert abs(f.std() - 0.02) < 2e-4 and abs(f.mean()) < 2e-4
    g = synth.layer_tensor("input_layernorm", seed=0)
    gf = (g.astype(np.uint32) << 16).view(np.float32)
    assert abs(gf.mean() - 1.0) < 0.01 and abs(gf.std() - 0.05) < 0.005


def test_adversarial_mix():
    w = synth.adversarial(1 << 22, seed=0)
    e = (w >> 7) & 0xFF
    m = w & 0x7F
    n = w.size
    zeros = np.count_nonzero((w & 0x7FFF) == 0)
    sub = np.count_nonzero((e == 0) & (m != 0))
    inf = np.count_nonzero((e == 0xFF) & (m == 0))
    nan = np.count_nonzero((e == 0xFF) & (m != 0))
    assert abs(zeros / n - 0.05) < 0.002
    assert 0.5e-4 < sub / n < 2e-4
    assert 10 < inf < 100 and 10 < nan < 100
    assert np.count_nonzero(w >> 15) > 0.4 * n  # both signs
    quiet = np.count_nonzero((e == 0xFF) & ((m & 0x40) != 0))
    assert 0 < quiet < nan  # quiet and signalling NaNs both present


def test_long_tail_mix():
    # N(0, 0.02) with 0.1 % of the weights moved to exponents across 1..254,
    # their sign and mantissa kept; deterministic per seed
    n = 1 << 20
    base = synth.normal(n, seed=4)
    w = synth.long_tail(n, seed=4)
    assert np.array_equal(w, synth.long_tail(n, seed=4))
    moved = np.flatnonzero(w != base)
    assert 0.8e-3 * n < moved.size <= 1e-3 * n
    assert np.array_equal(w[moved] & 0x807F, base[moved] & 0x807F)
    e = (w[moved] >> 7) & 0xFF
    assert e.min() >= 1 and e.max() <= 254 and np.unique(e).size > 200
