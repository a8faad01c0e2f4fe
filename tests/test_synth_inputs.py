"""The synthetic input recipe: seeded, deterministic, and distributed as follows.

Weights ~ N(0, 0.02) in bf16 (a normal truncated at 4.32 sigma by the 16-bit quantile table), norm
weights 1.0 (or bf16 draws of 1 + N(0, sigma^2) when asked for), ids uniform over the vocabulary, context lengths drawn from the stated set, prompt chunks
filled first-come-first-served up to the budget with only the last prompt cut, context K/V ~ N(0, 1).
"""
import numpy as np
from scipy import stats
from scipy.special import ndtri

import synth


def _bf16(bits):
    return synth.f32_from_bf16_bits(bits).astype(np.float64)


def test_weights_are_bf16_normal_draws_and_deterministic():
    s = synth.shape("tiny")
    w = synth.make_weights(s, seed=0)
    x = _bf16(w["model.layers.0.mlp.gate_proj.weight"])
    assert x.shape == (s.intermediate, s.hidden)
    np.testing.assert_array_equal(synth.bf16_bits_from_f32(x.astype(np.float32)),
                                  w["model.layers.0.mlp.gate_proj.weight"])          # bf16-exact
    assert abs(x.mean()) < 5e-4 and abs(x.std() - 0.02) < 5e-4
    edge = ndtri(65535.5 / 65536) * 0.02                                             # the table's last quantile
    assert np.abs(x).max() <= edge * (1 + 2.0 ** -8)                                 # plus its bf16 rounding
    assert stats.kstest(x.ravel()[::7] / 0.02, "norm").pvalue > 1e-3
    again = synth.make_weights(s, seed=0, cache=False)
    np.testing.assert_array_equal(again["model.layers.0.mlp.gate_proj.weight"],
                                  w["model.layers.0.mlp.gate_proj.weight"])           # regenerated alone
    other = synth.make_weights(s, seed=1)
    assert not np.array_equal(other["model.layers.0.mlp.gate_proj.weight"],
                              w["model.layers.0.mlp.gate_proj.weight"])
    assert not np.array_equal(w["model.layers.0.mlp.up_proj.weight"][:8], w["model.layers.0.mlp.gate_proj.weight"][:8])
    for name in ["model.norm.weight", "model.layers.1.input_layernorm.weight", "model.layers.0.self_attn.q_norm.weight"]:
        assert (_bf16(w[name]) == 1.0).all()


def test_ids_are_uniform_over_the_vocabulary():
    ids = synth.prompt_ids(200_000, 4096, key=3)
    assert ids.min() >= 0 and ids.max() < 4096
    counts = np.bincount(ids // 256, minlength=16)
    assert stats.chisquare(counts).pvalue > 1e-3
    np.testing.assert_array_equal(ids[:50], synth.prompt_ids(50, 4096, key=3)[:50])   # a prefix of the same stream


def test_context_lengths_come_from_the_stated_set():
    choices = (16, 64, 256, 1024, 4096)
    c = synth.context_lengths(20_000, choices, key=0, seed=0)
    assert set(np.unique(c).tolist()) == set(choices)
    assert stats.chisquare(np.array([(c == v).sum() for v in choices])).pvalue > 1e-3
    np.testing.assert_array_equal(synth.context_lengths(32, choices, key=0, seed=0),
                                  synth.context_lengths(32, choices, key=0, seed=0))


def test_prompt_chunk_is_filled_first_come_first_served():
    for key in range(20):
        chunk = synth.mixed_chunk_prompts(512, key=key, seed=0)
        assert sum(take for _, take in chunk) == 512
        assert all(p in (16, 64, 256, 1024, 4096) for p, _ in chunk)
        assert all(take == p for p, take in chunk[:-1])                   # only the last prompt is cut
        assert 0 < chunk[-1][1] <= chunk[-1][0]


def test_context_kv_is_standard_normal_bf16():
    s = synth.shape("qwen3_0p6b")
    kv = synth.kv_context(s, layer=3, request_key=7, ctx=300)
    assert kv.shape == (2, s.kv_heads, 300, s.head_dim)
    x = _bf16(kv)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    np.testing.assert_array_equal(kv, synth.kv_context(s, layer=3, request_key=7, ctx=300))
    assert not np.array_equal(kv, synth.kv_context(s, layer=4, request_key=7, ctx=300))


def test_random_norm_weights_are_one_plus_normal_draws():
    s = synth.shape("tiny")
    w = synth.make_weights(s, seed=0, norm_scale=0.1)
    names = ["model.norm.weight", "model.layers.0.input_layernorm.weight",
             "model.layers.0.post_attention_layernorm.weight", "model.layers.1.input_layernorm.weight",
             "model.layers.0.self_attn.q_norm.weight", "model.layers.0.self_attn.k_norm.weight"]
    vals = [_bf16(w[n]) for n in names]
    for n, x in zip(names, vals):
        np.testing.assert_array_equal(synth.bf16_bits_from_f32(x.astype(np.float32)), w[n])   # bf16-exact
        assert len(np.unique(x)) > x.size // 4                      # the entries differ from one another
    for i in range(len(vals)):
        for j in range(i + 1, len(vals)):
            if vals[i].shape == vals[j].shape:
                assert not np.array_equal(vals[i], vals[j])          # and from the other norms' weights
    big = np.concatenate([_bf16(synth.make_weights(synth.shape("qwen3_0p6b"), norm_scale=0.1)[
        f"model.layers.{l}.input_layernorm.weight"]) for l in range(8)])
    assert abs(big.mean() - 1.0) < 0.01 and abs(big.std() - 0.1) < 0.01
    assert stats.kstest((big[::3] - 1.0) / 0.1, "norm").pvalue > 1e-3
    # the matrices are the same draws as with unit norms
    np.testing.assert_array_equal(w["model.layers.0.mlp.down_proj.weight"],
                                  synth.make_weights(s, seed=0)["model.layers.0.mlp.down_proj.weight"])
