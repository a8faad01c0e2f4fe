"""Pins of the oracle's static-shape mixture-of-experts layer ("33. Removing overhead", §A MoE layer that
never asks the host): the grouping against brute-force invariants and a hand-worked case, the grouped
computation against the per-token definition, the definition against scalar loops and its algebraic
properties, and the router against a brute-force ranking."""
import math

import numpy as np
import pytest

import synth
from oracle import moe
from oracle.model import widen_bf16


def _brute_counts(flat, E):
    c = [0] * E
    for e in flat:
        c[int(e)] += 1
    return c


def test_moe_align_hand_worked():
    """Assignments 0..3 (tokens 0, 1 with two slots each) go to experts 2, 0, 0, 1; blocks of 2 rows."""
    sorted_ids, block_expert, num_padded = moe.moe_align(np.array([[2, 0], [0, 1]]), 3, 2)
    # expert 0: assignments 1, 2; expert 1: 3 and a padding row (4 = N * k); expert 2: 0 and padding;
    # room for 4 assignments + 3 * (2 - 1) padding rows, rounded to 8
    np.testing.assert_array_equal(sorted_ids, [1, 2, 3, 4, 0, 4, 4, 4])
    np.testing.assert_array_equal(block_expert, [0, 1, 2, 2])
    assert num_padded == 6


@pytest.mark.parametrize("N,k,E,bm", [(1, 1, 1, 16), (7, 2, 8, 16), (40, 8, 128, 16), (33, 2, 4, 64),
                                      (5, 8, 16, 4), (64, 8, 128, 64)])
def test_moe_align_invariants_on_random_routings(N, k, E, bm):
    rng = np.random.default_rng(N * 1000 + k * 10 + E)
    for trial in range(5):
        if trial == 0:
            ids = np.zeros((N, k), dtype=np.int64)                # everything on one expert
        else:
            ids = np.stack([rng.choice(E, size=k, replace=k > E) for _ in range(N)])
        flat = ids.reshape(-1)
        total = N * k
        sorted_ids, block_expert, num_padded = moe.moe_align(ids, E, bm)
        # static shapes: only N, k, E and bm decide them
        M = math.ceil((total + E * (bm - 1)) / bm) * bm
        assert sorted_ids.shape == (M,) and block_expert.shape == (M // bm,)
        counts = _brute_counts(flat, E)
        assert num_padded == sum(math.ceil(c / bm) * bm for c in counts) and num_padded % bm == 0
        real = sorted_ids[sorted_ids < total]
        assert sorted(real.tolist()) == list(range(total))       # every assignment exactly once
        assert (sorted_ids[num_padded:] == total).all()           # past the groups: padding only
        prev_e, prev_a = -1, -1
        for b in range(num_padded // bm):
            e = int(block_expert[b])
            assert e >= prev_e                                    # groups in expert order
            if e != prev_e:
                prev_a = -1
            rows = sorted_ids[b * bm:(b + 1) * bm]
            r = rows[rows < total]
            assert (flat[r] == e).all()                           # a block holds one expert's rows
            assert (np.diff(r) > 0).all() and (r.size == 0 or r[0] > prev_a)   # ascending (stable)
            if r.size:
                prev_a = int(r[-1])
            pads = np.flatnonzero(rows == total)                  # padding only at the end of a group
            assert pads.size == 0 or pads[0] == r.size
            prev_e = e
        assert (block_expert[num_padded // bm:] == E - 1).all()
        assert set(block_expert[:num_padded // bm].tolist()) == {e for e in range(E) if counts[e]}


def _tiny_layer(dtype="bf16"):
    m = synth.moe_shape("tiny_moe")
    w = synth.moe_weights(m, seed=0, dtype=dtype)
    x = widen_bf16(synth.moe_tokens(11, m.hidden, key=1))
    return m, x, widen_bf16(w["router"]), widen_bf16(w["gate_up"]), widen_bf16(w["down"])


@pytest.mark.parametrize("bm", [1, 2, 16, 64])
def test_grouped_layer_equals_the_per_token_definition(bm):
    m, x, wr, gu, dn = _tiny_layer()
    weights, ids = moe.route(x, wr, m.top_k)
    ref = moe.moe_reference(x, gu, dn, weights, ids)
    np.testing.assert_allclose(moe.moe_grouped(x, gu, dn, weights, ids, block_m=bm), ref, rtol=1e-12, atol=1e-15)


def test_per_token_definition_against_scalar_loops():
    rng = np.random.default_rng(3)
    N, D, I, E, k = 3, 4, 3, 3, 2
    x = rng.standard_normal((N, D))
    gu = rng.standard_normal((E, 2 * I, D))
    dn = rng.standard_normal((E, D, I))
    ids = np.array([[0, 2], [1, 0], [2, 1]])
    w = rng.random((N, k))
    want = np.zeros((N, D))
    for t in range(N):
        for j in range(k):
            e = ids[t, j]
            a = []
            for i in range(I):
                g = sum(gu[e, i, d] * x[t, d] for d in range(D))
                u = sum(gu[e, I + i, d] * x[t, d] for d in range(D))
                a.append(g / (1.0 + math.exp(-g)) * u)
            for d in range(D):
                want[t, d] += w[t, j] * sum(dn[e, d, i] * a[i] for i in range(I))
    np.testing.assert_allclose(moe.moe_reference(x, gu, dn, w, ids), want, rtol=1e-12)


def test_definition_is_linear_in_the_router_weights_and_blind_to_expert_labels():
    m, x, wr, gu, dn = _tiny_layer()
    weights, ids = moe.route(x, wr, m.top_k)
    base = moe.moe_reference(x, gu, dn, weights, ids)
    np.testing.assert_allclose(moe.moe_reference(x, gu, dn, 2.5 * weights, ids), 2.5 * base, rtol=1e-12)
    zero = weights.copy()
    zero[:, 1] = 0.0                                              # a zero weight removes that expert's share
    np.testing.assert_allclose(moe.moe_reference(x, gu, dn, zero, ids),
                               moe.moe_reference(x, gu, dn, weights[:, :1], ids[:, :1]), rtol=1e-12)
    perm = np.random.default_rng(0).permutation(m.experts)        # relabel the experts consistently
    inv = np.argsort(perm)
    np.testing.assert_allclose(moe.moe_reference(x, gu[perm], dn[perm], weights, inv[ids]), base, rtol=1e-12)


def test_router_ranking_and_weights():
    m, x, wr, _, _ = _tiny_layer()
    weights, ids = moe.route(x, wr, m.top_k)
    logits = x @ wr.T
    for t in range(x.shape[0]):
        ranked = sorted(range(m.experts), key=lambda e: (-logits[t, e], e))   # softmax is monotone
        assert ids[t].tolist() == ranked[:m.top_k]
    np.testing.assert_allclose(weights.sum(axis=1), 1.0, rtol=1e-12)
    # two experts, both chosen: the weights are the softmax itself, sigmoid of the logit difference
    xw = np.array([[1.0, -2.0]])
    wr2 = np.array([[0.3, 0.1], [-0.2, 0.4]])
    w2, i2 = moe.route(xw, wr2, 2)
    l0, l1 = xw[0] @ wr2[0], xw[0] @ wr2[1]
    assert i2[0].tolist() == [0, 1] and w2[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(l1 - l0)), rel=1e-12)
    # equal logits: the lower id first
    _, i3 = moe.route(np.zeros((1, 4)), np.ones((5, 4)), 3)
    assert i3[0].tolist() == [0, 1, 2]
