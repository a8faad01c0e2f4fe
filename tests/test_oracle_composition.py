"""Pins of the oracle's layer composition (forward_step), independent of the oracle itself.

1. Hand-worked logits (tests/golden/forward_handworked.json): two one-layer decoders with exact weights whose
   logits and final hidden states are derived by hand in closed form, following the layer order that
   "19. Fast decode", §Where the time goes, enumerates and SiLU on the gate half as in silu_and_mul
   ("33. Removing overhead", §Fewer, larger matmuls).
2. Special cases that reduce to library routines (torch's rms_norm and matrix products): with the output
   and down projections zero every layer is the identity, so the logits are the final norm of the
   embedding row times the embedding; and a request's first token (one key, at position 0) attends to its
   own value vector exactly, so with an identity output projection and a zero down projection the logits
   follow from v alone, with query head h reading KV head h // (q_heads / kv_heads).
3. Planted mistakes: each of the following, written into a copy of the oracle's source, makes at least one
   of the pins above fail -- SiLU on the up half, a dropped residual add (either one), the final norm
   skipped, QK-norm after RoPE, the input norm's weight used for the post-attention norm, a dropped QKV
   bias, attention that ignores the causal rule, RoPE rotating the other way, and the scale 1/d for 1/sqrt(d).
"""
from __future__ import annotations

import inspect
import json
import math
import os
import textwrap

import numpy as np
import pytest
import torch

import oracle
import oracle.model as om
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "forward_handworked.json")


def _bits(values) -> np.ndarray:
    x = np.asarray(values, dtype=np.float32)
    b = synth.bf16_bits_from_f32(x)
    assert np.array_equal(synth.f32_from_bf16_bits(b), x), "golden weights must be exact bf16 values"
    return b


def _golden_cases():
    g = json.load(open(GOLDEN))
    out = []
    for name, case in g["cases"].items():
        shape = synth.ModelShape(name="handworked_" + name, qkv_bias=case["qkv_bias"], **g["shape_common"])
        weights = {k: _bits(v) for k, v in case["weights"].items()}
        ns = {"sqrt": math.sqrt, "exp": math.exp, "cos": math.cos, "sin": math.sin}
        for var, expr in case["defs"]:
            ns[var] = float(eval(expr, {"__builtins__": {}}, ns))
        logits = np.array([float(eval(e, {"__builtins__": {}}, ns)) for e in case["logits"]])
        hidden = np.array([[float(eval(e, {"__builtins__": {}}, ns)) for e in row] for row in case["hidden"]])
        out.append((name, shape, weights, case["token_ids"], case["positions"], logits, hidden))
    return out


def _run(fwd, shape, weights, ids, pos):
    model = oracle.OracleModel(shape, weights)
    cache = oracle.ContiguousCache(shape, {0: 8})
    logits, h = fwd(model, cache, ids, pos, [0, len(ids)], return_hidden=True)
    return logits[0], h


def _golden_holds(fwd=None) -> bool:
    fwd = fwd or om.forward_step
    for name, shape, weights, ids, pos, want_logits, want_hidden in _golden_cases():
        logits, h = _run(fwd, shape, weights, ids, pos)
        if not (np.allclose(logits, want_logits, rtol=0, atol=1e-12) and
                np.allclose(h[-len(want_hidden):], want_hidden, rtol=0, atol=1e-12)):
            return False
    return True


@pytest.mark.parametrize("attention", ["split", "rows", "packed"])
def test_forward_matches_hand_worked_logits(attention):
    for name, shape, weights, ids, pos, want_logits, want_hidden in _golden_cases():
        model = oracle.OracleModel(shape, weights)
        cache = oracle.ContiguousCache(shape, {0: 8})
        logits, h = oracle.forward_step(model, cache, ids, pos, [0, len(ids)], attention=attention,
                                        return_hidden=True)
        np.testing.assert_allclose(logits[0], want_logits, rtol=0, atol=1e-12, err_msg=name)
        np.testing.assert_allclose(h, want_hidden, rtol=0, atol=1e-12, err_msg=name)


# ----------------------------------------------------------------------------- special cases


class _Override:
    """Synthetic weights with some tensors replaced (uint16 bf16 bits)."""

    def __init__(self, base, repl: dict):
        self.base, self.repl = base, repl

    def __getitem__(self, name):
        return self.repl[name] if name in self.repl else self.base[name]

    def __contains__(self, name):
        return name in self.base


def _f(bits) -> torch.Tensor:
    return torch.from_numpy(oracle.widen_bf16(bits))


def test_zero_output_and_down_projections_leave_the_embedding_row():
    s = synth.shape("tiny")
    base = synth.make_weights(s, seed=2, norm_scale=0.1)
    zero = {}
    for l in range(s.layers):
        zero[f"model.layers.{l}.self_attn.o_proj.weight"] = np.zeros((s.hidden, s.q_size), np.uint16)
        zero[f"model.layers.{l}.mlp.down_proj.weight"] = np.zeros((s.hidden, s.intermediate), np.uint16)
    w = _Override(base, zero)
    ids = synth.prompt_ids(5, s.vocab, 9)
    model = oracle.OracleModel(s, w)
    logits = oracle.forward_step(model, oracle.ContiguousCache(s, {0: 8}), ids, np.arange(5), [0, 5])
    E = _f(base["model.embed_tokens.weight"])
    y = torch.nn.functional.rms_norm(E[int(ids[-1])], (s.hidden,), weight=_f(base["model.norm.weight"]), eps=s.rms_eps)
    np.testing.assert_allclose(logits[0], (E @ y).numpy(), rtol=0, atol=1e-10)


def test_first_token_attends_to_its_own_value_vector():
    # hidden == q_heads * head_dim so that the output projection can be the identity
    s = synth.ModelShape("first_token", layers=1, hidden=128, q_heads=4, kv_heads=2, head_dim=32, intermediate=64,
                         vocab=512, qk_norm=True, qkv_bias=True, tie_embeddings=True)
    base = synth.make_weights(s, seed=3, norm_scale=0.1)
    eye = synth.bf16_bits_from_f32(np.eye(s.hidden, dtype=np.float32))
    w = _Override(base, {"model.layers.0.self_attn.o_proj.weight": eye,
                         "model.layers.0.mlp.down_proj.weight": np.zeros((s.hidden, s.intermediate), np.uint16)})
    E = _f(base["model.embed_tokens.weight"])
    for tok in (0, 7, 300):
        model = oracle.OracleModel(s, w)
        logits = oracle.forward_step(model, oracle.ContiguousCache(s, {0: 4}), [tok], [0], [0, 1])
        x = torch.nn.functional.rms_norm(E[tok], (s.hidden,), weight=_f(base["model.layers.0.input_layernorm.weight"]),
                                         eps=s.rms_eps)
        v = _f(base["model.layers.0.self_attn.v_proj.weight"]) @ x + _f(base["model.layers.0.self_attn.v_proj.bias"])
        v = v.reshape(s.kv_heads, s.head_dim)
        o = torch.cat([v[h // (s.q_heads // s.kv_heads)] for h in range(s.q_heads)])
        h_out = E[tok] + o
        y = torch.nn.functional.rms_norm(h_out, (s.hidden,), weight=_f(base["model.norm.weight"]), eps=s.rms_eps)
        np.testing.assert_allclose(logits[0], (E @ y).numpy(), rtol=0, atol=1e-10)


# ----------------------------------------------------------------------------- planted mistakes


def _mutant(func, old: str, new: str):
    """A copy of one oracle function with `old` replaced by `new` in its source (old must occur once)."""
    src = textwrap.dedent(inspect.getsource(func))
    assert src.count(old) == 1, f"mutation anchor not found once in {func.__name__}: {old!r}"
    ns = dict(om.__dict__)
    exec(compile(src.replace(old, new), f"<mutant of {func.__name__}>", "exec"), ns)
    return ns[func.__name__]


_QK_BEFORE = '''        if s.qk_norm:
            q = rms_norm(q, model.get(p + "self_attn.q_norm.weight"), s.rms_eps)
            k = rms_norm(k, model.get(p + "self_attn.k_norm.weight"), s.rms_eps)
        q = apply_rope(q, positions, s.rope_theta)
        k = apply_rope(k, positions, s.rope_theta)
'''
_QK_AFTER = '''        q = apply_rope(q, positions, s.rope_theta)
        k = apply_rope(k, positions, s.rope_theta)
        if s.qk_norm:
            q = rms_norm(q, model.get(p + "self_attn.q_norm.weight"), s.rms_eps)
            k = rms_norm(k, model.get(p + "self_attn.k_norm.weight"), s.rms_eps)
'''

FORWARD_MUTATIONS = {
    "silu on the up half": ("act(silu(g) * u)", "act(g * silu(u))"),
    "attention residual dropped": ("h = h + act(o.reshape(T, s.q_size))", "h = act(o.reshape(T, s.q_size))"),
    "MLP residual dropped": ("h = h + act(silu(g) * u)", "h = act(silu(g) * u)"),
    "final norm skipped": ('y = act(rms_norm(h[last], model.get("model.norm.weight"), s.rms_eps))', "y = act(h[last])"),
    "QK-norm after RoPE": (_QK_BEFORE, _QK_AFTER),
    "input norm weight for the post-attention norm": ('p + "post_attention_layernorm.weight"', 'p + "input_layernorm.weight"'),
    "QKV bias dropped": ('v = v + model.get(p + "self_attn.v_proj.bias")', "v = v"),
}

HELPER_MUTATIONS = {
    "causal rule ignored": (om.attend_packed, "mask = kpos[None, :] <= positions[:, None]", "mask = kpos[None, :] >= 0"),
    "RoPE rotating the other way": (om.apply_rope, "[x1 * cos - x2 * sin, x2 * cos + x1 * sin]",
                                    "[x1 * cos + x2 * sin, x2 * cos - x1 * sin]"),
    "scale 1/d": (om.attend_packed, "scale = 1.0 / np.sqrt(s.head_dim)", "scale = 1.0 / s.head_dim"),
}


def test_unmutated_copy_still_holds():
    assert _golden_holds(_mutant(om.forward_step, "act(silu(g) * u)", "act(silu(g) * u)"))


@pytest.mark.parametrize("name", sorted(FORWARD_MUTATIONS))
def test_planted_mistake_in_the_layer_is_caught(name):
    old, new = FORWARD_MUTATIONS[name]
    assert not _golden_holds(_mutant(om.forward_step, old, new)), name


@pytest.mark.parametrize("name", sorted(HELPER_MUTATIONS))
def test_planted_mistake_in_a_helper_is_caught(name, monkeypatch):
    func, old, new = HELPER_MUTATIONS[name]
    monkeypatch.setattr(om, func.__name__, _mutant(func, old, new))
    assert not _golden_holds(), name
