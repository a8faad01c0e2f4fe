"""Pins of the oracle's IEEE binary16 pieces: the fp16 variant of a model (fp16 weights, activations and cache).

The bf16 path's counterparts are pinned in test_oracle_math.py.  Here the format's decoding is checked
exhaustively, the rounding against numpy's float64 -> float16 conversion (a library routine) on every
tie and on random values across the whole range, and the fp16 forward against the float64 forward.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle.model import F16_MAX


def test_widen_f16_decodes_every_pattern_like_numpy():
    bits = np.arange(65536, dtype=np.uint64).astype(np.uint16)
    ours = oracle.widen_f16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()
    assert np.signbit(ours[0x8000]) and ours[0x8000] == 0.0                 # -0
    assert ours[0x0001] == 2.0 ** -24 and ours[0x7BFF] == F16_MAX          # smallest subnormal, largest finite


def test_round_f16_is_the_identity_on_fp16_values():
    bits = np.arange(65536, dtype=np.uint64).astype(np.uint16)
    v = oracle.widen_f16(bits)
    fin = np.isfinite(v)
    np.testing.assert_array_equal(oracle.round_f16(v[fin]), v[fin])


def test_round_f16_ties_go_to_even_at_every_midpoint():
    """The exact midpoint between each pair of neighbouring positive fp16 values (exact in float64)."""
    v = oracle.widen_f16(np.arange(0, 0x7C00, dtype=np.uint64).astype(np.uint16))   # 0 .. 65504
    mid = (v[:-1] + v[1:]) / 2
    ours = oracle.round_f16(mid)
    with np.errstate(over="ignore"):
        ref = mid.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(ours, ref)
    even = np.arange(len(mid)) % 2 == 0                                    # pattern k even: the tie goes down
    np.testing.assert_array_equal(ours[even], v[:-1][even])
    np.testing.assert_array_equal(ours[~even], v[1:][~even])
    # one float64 ulp either side of a midpoint decides by distance
    np.testing.assert_array_equal(oracle.round_f16(np.nextafter(mid, 0)), v[:-1])
    np.testing.assert_array_equal(oracle.round_f16(np.nextafter(mid, np.inf)), v[1:])


def test_round_f16_matches_numpy_across_the_range():
    rng = np.random.default_rng(12)
    mag = np.exp2(rng.uniform(-27, 17, size=2_000_000))
    x = mag * np.where(rng.random(mag.size) < 0.5, -1.0, 1.0)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(oracle.round_f16(x), ref)
    assert oracle.round_f16(np.array([65519.99]))[0] == F16_MAX              # rounds down to the largest
    assert oracle.round_f16(np.array([65520.0]))[0] == np.inf                # the tie past it overflows
    assert oracle.round_f16(np.array([2.0 ** -25]))[0] == 0.0                # tie between 0 and 2^-24: even


def test_synthetic_fp16_weights_are_the_bf16_draws_in_the_other_format():
    s = synth.shape("tiny")
    wf, wb = synth.make_weights(s, dtype="f16"), synth.make_weights(s)
    for name in ["model.layers.0.self_attn.q_proj.weight", "model.layers.1.mlp.down_proj.weight"]:
        a = oracle.widen_f16(wf[name])
        b = oracle.widen_bf16(wb[name])
        np.testing.assert_array_equal(oracle.round_f16(a), a)              # fp16-exact
        # the same quantile, rounded to 11 and to 8 significant bits
        assert np.all(np.abs(a - b) <= np.abs(b) * (2.0 ** -8 + 2.0 ** -11) + 2.0 ** -24)
        assert abs(a.std() - 0.02) < 0.002 and abs(a.mean()) < 0.002
    assert (oracle.widen_f16(wf["model.norm.weight"]) == 1.0).all()
    kv = synth.kv_context(s, 0, 3, 40, dtype="f16")
    kb = synth.kv_context(s, 0, 3, 40)
    assert np.all(np.abs(oracle.widen_f16(kv) - oracle.widen_bf16(kb)) <= np.abs(oracle.widen_bf16(kb)) * 2.0 ** -7)


def test_fp16_step_stays_near_the_float64_forward():
    """Tiny shape with fp16 weights: rounding the activations and the cache to fp16 moves the logits by
    far less than rounding them to bf16 does (11 against 8 significant bits), and both stay close."""
    s = synth.shape("tiny")
    wf = synth.make_weights(s, dtype="f16")
    model = oracle.OracleModel(s, wf, dtype="f16")
    P = 16
    ids = np.concatenate([synth.prompt_ids(P, s.vocab, r) for r in range(2)])
    pos = np.concatenate([np.arange(P)] * 2)
    cu = [0, P, 2 * P]
    out = {}
    for mode in ["f64", "f16", "bf16"]:
        cache = oracle.ContiguousCache(s, {0: P, 1: P})
        out[mode] = oracle.forward_step(model, cache, ids, pos, cu, activations=mode)
    e16 = np.abs(out["f16"] - out["f64"]).max()
    eb = np.abs(out["bf16"] - out["f64"]).max()
    assert 0 < e16 < 0.02 and e16 < eb / 3, (e16, eb)
    with pytest.raises(ValueError):
        oracle.OracleModel(s, wf, dtype="f32")
