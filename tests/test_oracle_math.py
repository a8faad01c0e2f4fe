"""Pins of the oracle's forward pieces against closed forms, library routines and brute force."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import model as om

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------- RMSNorm, SiLU


def test_rms_norm_matches_torch_library():
    x = RNG.standard_normal((7, 96))
    w = RNG.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, w, 1e-6), ref, rtol=1e-13, atol=1e-13)


def test_rms_norm_constant_vector_closed_form():
    c, eps = -3.25, 1e-6
    w = np.linspace(0.5, 2.0, 64)
    out = oracle.rms_norm(np.full((1, 64), c), w, eps)
    np.testing.assert_allclose(out[0], c / np.sqrt(c * c + eps) * w, rtol=1e-15)


def test_silu_matches_torch_library():
    g = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(oracle.silu(g), torch.nn.functional.silu(torch.from_numpy(g)).numpy(),
                               rtol=1e-14, atol=1e-300)


# ----------------------------------------------------------------------------- RoPE


def test_rope_identity_at_position_zero():
    x = RNG.standard_normal((3, 4, 64))
    np.testing.assert_array_equal(oracle.apply_rope(x, np.zeros(3), 1e6), x)


def test_rope_preserves_norm():
    x = RNG.standard_normal((5, 2, 128))
    y = oracle.apply_rope(x, np.array([1, 17, 300, 4095, 70000]), 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_dot_depends_on_relative_position_only():
    q = RNG.standard_normal((1, 1, 64))
    k = RNG.standard_normal((1, 1, 64))
    dots = []
    for m, n in [(10, 3), (107, 100), (5007, 5000)]:
        qm = oracle.apply_rope(q, np.array([m]), 1e4)
        kn = oracle.apply_rope(k, np.array([n]), 1e4)
        dots.append(float((qm * kn).sum()))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


def test_rope_d2_is_complex_rotation():
    x = np.array([[[0.3, -1.7]]])
    for pos in [0, 1, 5, 123]:
        y = oracle.apply_rope(x, np.array([pos]), 1e6)
        z = complex(0.3, -1.7) * np.exp(1j * pos)          # d = 2: inv_freq = theta^0 = 1
        np.testing.assert_allclose([y[0, 0, 0], y[0, 0, 1]], [z.real, z.imag], rtol=1e-13, atol=1e-15)


def test_rope_pairs_rotate_half_with_theta_powers():
    # d = 4: pair (x0, x2) turns by pos * theta^0, pair (x1, x3) by pos * theta^(-1/2).
    theta = 1e6
    x = RNG.standard_normal((1, 1, 4))
    pos = 7
    y = oracle.apply_rope(x, np.array([pos]), theta)[0, 0]
    for i, f in [(0, 1.0), (1, theta ** -0.5)]:
        z = complex(x[0, 0, i], x[0, 0, i + 2]) * np.exp(1j * pos * f)
        np.testing.assert_allclose([y[i], y[i + 2]], [z.real, z.imag], rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------- attention


def _brute_attention(q, K, V, scale):
    """Softmax attention with Python loops and math.exp only (tiny inputs)."""
    import math
    n = len(K)
    s = [sum(q[j] * K[i][j] for j in range(len(q))) * scale for i in range(n)]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    tot = sum(e)
    return [sum(e[i] / tot * V[i][j] for i in range(n)) for j in range(len(V[0]))]


def test_attend_one_matches_brute_force():
    q = RNG.standard_normal(8)
    K = RNG.standard_normal((5, 8))
    V = RNG.standard_normal((5, 8))
    ref = _brute_attention(q.tolist(), K.tolist(), V.tolist(), 1 / np.sqrt(8))
    np.testing.assert_allclose(oracle.attend_one(q, K, V, 1 / np.sqrt(8)), ref, rtol=1e-12)


def _tiny_shape(q_heads=4, kv_heads=2, d=16):
    return synth.ModelShape("t", layers=1, hidden=32, q_heads=q_heads, kv_heads=kv_heads, head_dim=d,
                            intermediate=64, vocab=50)


@pytest.mark.parametrize("q_heads,kv_heads", [(4, 2), (6, 2), (4, 4), (8, 1)])
def test_packed_attention_matches_torch_sdpa_with_gqa(q_heads, kv_heads):
    s = _tiny_shape(q_heads, kv_heads)
    n = 11
    cache = oracle.ContiguousCache(s, {0: 32})
    k = RNG.standard_normal((n, kv_heads, 16))
    v = RNG.standard_normal((n, kv_heads, 16))
    q = RNG.standard_normal((n, q_heads, 16))
    pos = np.arange(n)
    cache.write(0, 0, pos, k, v)
    out = oracle.attend_packed(s, cache, 0, q, 0, pos)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]                     # [1, H, n, d]
    group = q_heads // kv_heads
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(group, dim=0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(group, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_rows_equal_packed_and_paged_equals_contiguous():
    s = _tiny_shape(4, 2)
    n = 37
    k = RNG.standard_normal((n, 2, 16))
    v = RNG.standard_normal((n, 2, 16))
    q = RNG.standard_normal((n, 4, 16))
    pos = np.arange(n)
    contiguous = oracle.ContiguousCache(s, {0: 64})
    contiguous.write(0, 0, pos, k, v)
    paged = oracle.PagedCache(s, num_blocks=16, block_size=16)
    paged.set_block_table(0, [11, 3, 7])                                 # permuted blocks
    paged.write(0, 0, pos, k, v)
    rows_c = oracle.attend_rows(s, contiguous, 0, q, [0] * n, pos)
    rows_p = oracle.attend_rows(s, paged, 0, q, [0] * n, pos)
    np.testing.assert_array_equal(rows_c, rows_p)                         # same keys, same arithmetic
    packed = oracle.attend_packed(s, paged, 0, q, 0, pos)
    np.testing.assert_allclose(packed, rows_p, rtol=1e-12, atol=1e-13)


def test_padding_row_outputs_zero_and_leaves_real_rows_alone():
    s = _tiny_shape(4, 2)
    cache = oracle.PagedCache(s, num_blocks=4)
    cache.set_block_table(0, [2])
    k = RNG.standard_normal((5, 2, 16))
    v = RNG.standard_normal((5, 2, 16))
    cache.write(0, 0, np.arange(5), k, v)
    q = RNG.standard_normal((2, 4, 16))
    alone = oracle.attend_rows(s, cache, 0, q[:1], [0], [4])
    padded = oracle.attend_rows(s, cache, 0, q, [0, None], [4, 0])
    np.testing.assert_array_equal(padded[0], alone[0])
    np.testing.assert_array_equal(padded[1], 0.0)


def test_paged_slot_mapping_and_scratch_block():
    s = _tiny_shape()
    cache = oracle.PagedCache(s, num_blocks=8, block_size=16)
    cache.set_block_table(0, [5, 2])
    assert cache.slot(0, 0) == 80 and cache.slot(0, 15) == 95 and cache.slot(0, 16) == 32
    assert cache.slot(None, 0) == -1
    cache.write_slot(0, -1, np.ones((2, 16)), np.ones((2, 16)))
    np.testing.assert_array_equal(cache.block_contents(0, 8)[:, :, 0, :], 1.0)   # scratch = num_blocks
    with pytest.raises(ValueError):
        cache.slot(0, 32)


# ----------------------------------------------------------------------------- fusion


def test_fused_projections_equal_separate():
    x = RNG.standard_normal((9, 64))
    wq, wk, wv = RNG.standard_normal((96, 64)), RNG.standard_normal((32, 64)), RNG.standard_normal((32, 64))
    fused = x @ oracle.fused_qkv(wq, wk, wv).T
    np.testing.assert_allclose(fused, np.concatenate([x @ wq.T, x @ wk.T, x @ wv.T], axis=1), rtol=1e-13,
                               atol=1e-13)
    wg, wu = RNG.standard_normal((80, 64)), RNG.standard_normal((80, 64))
    gu = x @ oracle.fused_gate_up(wg, wu).T
    np.testing.assert_allclose(gu, np.concatenate([x @ wg.T, x @ wu.T], axis=1), rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- whole step properties


def _tiny_model():
    s = synth.shape("tiny")
    return s, oracle.OracleModel(s, synth.make_weights(s, seed=0))


def _paged(s, tables, nb=64):
    c = oracle.PagedCache(s, nb)
    for r, t in tables.items():
        c.set_block_table(r, t)
    return c


def test_step_attention_split_equals_rows_and_packed():
    s, m = _tiny_model()
    p0 = synth.prompt_ids(20, s.vocab, 0)
    p1 = synth.prompt_ids(9, s.vocab, 1)
    ids = np.concatenate([p0, p1])
    pos = np.concatenate([np.arange(20), np.arange(9)])
    cu = np.array([0, 20, 29])
    outs = []
    for mode in ["split", "rows", "packed"]:
        c = _paged(s, {0: [0, 1], 1: [2]})
        outs.append(oracle.forward_step(m, c, ids, pos, cu, attention=mode))
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(outs[0], outs[2], rtol=1e-10, atol=1e-11)


def test_step_requests_are_independent():
    s, m = _tiny_model()
    p0 = synth.prompt_ids(16, s.vocab, 0)
    p1 = synth.prompt_ids(16, s.vocab, 1)
    both = oracle.forward_step(m, _paged(s, {0: [0], 1: [1]}), np.concatenate([p0, p1]),
                               np.concatenate([np.arange(16)] * 2), [0, 16, 32])
    alone = oracle.forward_step(m, _paged(s, {0: [4]}), p1, np.arange(16), [0, 16])
    np.testing.assert_allclose(both[1], alone[0], rtol=1e-11, atol=1e-11)


def test_incremental_decode_equals_full_prefill():
    """Prefill 16 + two decode steps (chunked, cached keys) equals one prefill of 18 tokens."""
    s, m = _tiny_model()
    ids = synth.prompt_ids(18, s.vocab, 7)
    c = _paged(s, {0: [3, 9]})
    oracle.forward_step(m, c, ids[:10], np.arange(10), [0, 10])           # chunk 1
    oracle.forward_step(m, c, ids[10:16], np.arange(10, 16), [0, 6])      # chunk 2
    oracle.forward_step(m, c, ids[16:17], [16], [0, 1])                   # decode
    step = oracle.forward_step(m, c, ids[17:18], [17], [0, 1])            # decode
    full = oracle.forward_step(m, _paged(s, {0: [0, 1]}), ids, np.arange(18), [0, 18])
    np.testing.assert_allclose(step, full, rtol=1e-10, atol=1e-10)


def test_step_paged_equals_contiguous_cache():
    s, m = _tiny_model()
    ids = synth.prompt_ids(21, s.vocab, 3)
    a = oracle.forward_step(m, _paged(s, {0: [6, 1]}), ids, np.arange(21), [0, 21], attention="rows")
    b = oracle.forward_step(m, oracle.ContiguousCache(s, {0: 40}), ids, np.arange(21), [0, 21],
                            attention="rows")
    np.testing.assert_array_equal(a, b)


def test_planted_mistake_is_caught(monkeypatch):
    """A wrong GQA head mapping in the oracle must break the torch SDPA pin."""
    s = _tiny_shape(4, 2)
    cache = oracle.ContiguousCache(s, {0: 16})
    n = 6
    k = RNG.standard_normal((n, 2, 16))
    v = RNG.standard_normal((n, 2, 16))
    q = RNG.standard_normal((n, 4, 16))
    cache.write(0, 0, np.arange(n), k, v)
    good = oracle.attend_rows(s, cache, 0, q, [0] * n, np.arange(n))

    def wrong_rows(s_, cache_, layer, q_, reqs, positions):
        out = np.zeros_like(q_)
        for i, (r, p) in enumerate(zip(reqs, positions)):
            K, V, kpos = cache_.read(layer, r, int(p) + 1)
            vis = kpos <= int(p)
            for h in range(s_.q_heads):
                g = h % s_.kv_heads                                          # planted: modulo instead of //
                out[i, h] = oracle.attend_one(q_[i, h], K[g][vis], V[g][vis], 1 / np.sqrt(s_.head_dim))
        return out

    bad = wrong_rows(s, cache, 0, q, [0] * n, np.arange(n))
    assert not np.allclose(good, bad)


# ----------------------------------------------------------------------------- bf16 activations


def test_round_bf16_matches_torch_on_float32_values():
    """Every float32 value has one nearest bf16 value: torch's conversion is the library pin, with
    exact ties (low 16 bits 0x8000) of both significand parities included."""
    x32 = (RNG.standard_normal(200000) * np.exp2(RNG.integers(-30, 30, 200000))).astype(np.float32)
    bits = RNG.integers(0x00800000, 0x7F000000, 4000, dtype=np.uint32)
    ties = ((bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    x32 = np.concatenate([x32, ties, -ties])
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(om.round_bf16(x32.astype(np.float64)), want)


def test_round_bf16_is_nearest_with_ties_to_even_brute_force():
    """Float64 inputs (no float32 step in between): the nearest of all bf16 values in [1/4, 4] by
    exhaustive search, an exact midpoint going to the even bit pattern."""
    grid_bits = np.arange(0x3E80, 0x4081, dtype=np.uint16)
    grid = om.widen_bf16(grid_bits)
    mids = (grid[:-1] + grid[1:]) / 2
    x = np.concatenate([RNG.uniform(0.2501, 3.999, 3000), mids[::5], grid[::11]])
    got = om.round_bf16(x)
    for xi, gi in zip(x, got):
        d = np.abs(grid - xi)
        near = np.flatnonzero(d == d.min())
        pick = near[0] if len(near) == 1 else next(i for i in near if grid_bits[i] % 2 == 0)
        assert gi == grid[pick], (xi, gi, grid[pick])
    np.testing.assert_array_equal(om.round_bf16(-x), -got)


def test_bf16_activation_step_caches_bf16_values_and_stays_near_f64():
    s, m = _tiny_model()
    ids = synth.prompt_ids(21, s.vocab, 3)
    c64, c16 = oracle.ContiguousCache(s, {0: 40}), oracle.ContiguousCache(s, {0: 40})
    a = oracle.forward_step(m, c64, ids, np.arange(21), [0, 21])
    b = oracle.forward_step(m, c16, ids, np.arange(21), [0, 21], activations="bf16")
    assert 0 < np.abs(a - b).max() < 0.05
    for l in range(s.layers):
        for kv in (c16.keys[(l, 0)][:, :21], c16.values[(l, 0)][:, :21]):
            np.testing.assert_array_equal(om.round_bf16(kv), kv)                # the cache holds bf16 values
        assert not np.array_equal(om.round_bf16(c64.keys[(l, 0)][:, :21]), c64.keys[(l, 0)][:, :21])
    with pytest.raises(ValueError):
        oracle.forward_step(m, c16, ids[:1], [21], [0, 1], activations="fp16")
