"""Pins of the oracle's top-k / top-p filters and of its float32 exp.

"19. Fast decode", §Sampling without the CPU: top-k and top-p filters set the dropped logits to -inf
before the Gumbel-max argmax.  The pins below do not restate the oracle: they use libm, exact integer
distributions whose nucleus is known in closed form, brute force over prefixes, torch.topk, the pinned
unfiltered sampler, and chi-squared tests of the draws against the filtered softmax.
"""
import math

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import filters as fl
from oracle import sampler as osm


def test_exp_f32_within_two_ulp_of_libm_on_its_range():
    lo = int(np.array([-23.0], dtype=np.float32).view(np.uint32)[0])
    bits = np.arange(0x80000000, lo + 1, 101, dtype=np.uint64).astype(np.uint32)
    d = bits.view(np.float32)
    e = fl.exp_f32(d)
    exact = np.exp(d.astype(np.float64))
    ulp = np.spacing(e.astype(np.float32)).astype(np.float64)
    assert (np.abs(e.astype(np.float64) - exact) / ulp).max() <= 2.0


def test_exp_f32_special_points():
    assert fl.exp_f32(np.float32(0.0)) == np.float32(1.0)
    assert fl.exp_f32(np.float32(-0.0)) == np.float32(1.0)
    out = fl.exp_f32(np.array([-math.log(2.0), -1.0, -10.0], dtype=np.float32)).astype(np.float64)
    np.testing.assert_allclose(out, [0.5, math.exp(-1.0), math.exp(-10.0)], rtol=2 ** -22)
    np.testing.assert_array_equal(fl.exp_f32(np.array([-23.5, -100.0, -1e30], dtype=np.float32)), 0.0)
    # below -23 the weight floor(e * 2^32) is 0 whatever the value: exp(-23) < 2^-32
    assert math.exp(-23.0) * 2 ** 32 < 1.0


def _shortest_prefix(w, P):
    """Brute force: the shortest prefix whose mass reaches P / 2^24 of the total (exact integers)."""
    W = sum(w)
    for n in range(1, len(w) + 1):
        if sum(w[:n]) * 2 ** 24 >= P * W:
            return n
    return len(w)


def test_nucleus_size_matches_brute_force_shortest_prefix():
    rng = np.random.default_rng(3)
    for _ in range(400):
        n = int(rng.integers(1, 12))
        w = [int(x) for x in rng.integers(0, 2 ** 32 + 1, size=n)]
        w[0] = 2 ** 32                                       # the top entry always has weight 2^32
        if rng.random() < 0.3:
            w = [w[0]] + [int(x) for x in rng.integers(0, 4, size=n - 1)]   # tiny tails, zero weights
        P = int(rng.integers(1, 2 ** 24))
        assert fl.nucleus_size(np.array(w, dtype=np.int64), P) == _shortest_prefix(w, P)


def test_nucleus_boundary_in_closed_form():
    """Masses 1/2, 1/4, 1/8, 1/8: p = 3/4 is reached exactly by two entries; one unit more needs three."""
    w = np.array([2 ** 32, 2 ** 31, 2 ** 30, 2 ** 30], dtype=np.int64)
    assert fl.nucleus_size(w, 3 * 2 ** 22) == 2
    assert fl.nucleus_size(w, 3 * 2 ** 22 + 1) == 3
    assert fl.nucleus_size(w, 2 ** 23) == 1                  # p = 1/2: the top entry alone reaches it
    assert fl.nucleus_size(w, 1) == 1                        # the smallest p keeps the top entry
    assert fl.nucleus_size(w, 2 ** 24 - 1) == 4


def test_p_units():
    assert fl.p_units(0.75) == 3 * 2 ** 22
    assert fl.p_units(1.0) == 0 and fl.p_units(0.0) == 0 and fl.p_units(-0.5) == 0 and fl.p_units(2.0) == 0
    assert fl.p_units(1e-12) == 1                            # rounds to 0 units, kept at 1
    assert fl.p_units(1.0 - 2 ** -26) == 0                   # rounds to 2^24 units: no filter


def test_rank_order_ties_and_signed_zero():
    z = np.array([1.0, 3.0, 1.0, -0.0, 0.0, 3.0], dtype=np.float32)
    np.testing.assert_array_equal(fl.rank_order(z), [1, 5, 0, 2, 3, 4])
    np.testing.assert_array_equal(fl.survivors(np.array([-0.0, 0.0, -1.0], dtype=np.float32), 1.0, 1, 1.0), [0])
    np.testing.assert_array_equal(fl.survivors(np.array([1, 1, 1, 0], dtype=np.float32), 1.0, 2, 1.0), [0, 1])


def test_top_k_set_matches_torch_topk_on_distinct_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    for trial in range(30):
        V = int(rng.integers(2, 3000))
        z = rng.permutation(V).astype(np.float32) * np.float32(0.01) - np.float32(3.0)   # distinct values
        k = int(rng.integers(1, V + 1))
        ref = np.sort(torch.topk(torch.from_numpy(z), k).indices.numpy())
        np.testing.assert_array_equal(fl.survivors(z, 0.9, k, 1.0), ref)


def test_top_p_nucleus_of_a_dyadic_distribution():
    """Softmax masses 8:4:2:1:1 (/16): cumulative 0.5, 0.75, 0.875, 0.9375, 1."""
    z = np.log(np.array([1, 8, 2, 4, 1], dtype=np.float64)).astype(np.float32)  # ranked: 1, 3, 2, 0, 4
    for p, want in [(0.3, [1]), (0.6, [1, 3]), (0.8, [1, 2, 3]), (0.9, [0, 1, 2, 3]), (0.99, [0, 1, 2, 3, 4])]:
        np.testing.assert_array_equal(fl.survivors(z, 1.0, 0, p), want)
    # temperature 0.5 squares the masses: 64:16:4:1:1 (/86) -> cumulative 0.744, 0.930, ...
    np.testing.assert_array_equal(fl.survivors(z, 0.5, 0, 0.9), [1, 3])
    np.testing.assert_array_equal(fl.survivors(z, 0.5, 0, 0.95), [1, 2, 3])


def test_top_p_renormalises_over_the_top_k_survivors():
    z = np.zeros(8, dtype=np.float32)                        # eight equal masses
    np.testing.assert_array_equal(fl.survivors(z, 1.0, 4, 0.5), [0, 1])      # 1/4 each among four
    np.testing.assert_array_equal(fl.survivors(z, 1.0, 0, 0.5), [0, 1, 2, 3])  # 1/8 each among eight


def test_special_cases_reduce_to_the_unfiltered_sampler_and_argmax():
    rng = np.random.default_rng(11)
    for row in range(12):
        V = int(rng.integers(2, 5000))
        z = (rng.standard_normal(V) * 2.0).astype(np.float32)
        T = [0.6, 1.0, 1.7][row % 3]
        plain = oracle.sample_row(z, T, 5, row, row)
        assert fl.sample_row_filtered(z, T, 0, 1.0, 5, row, row) == plain
        assert fl.sample_row_filtered(z, T, V, 0.0, 5, row, row) == plain
        assert fl.sample_row_filtered(z, T, V + 3, 1.5, 5, row, row) == plain
        assert fl.sample_row_filtered(z, T, 1, 0.9, 5, row, row) == int(np.argmax(z))
        assert fl.sample_row_filtered(z, T, 0, 1e-9, 5, row, row) == int(np.argmax(z))
        assert fl.sample_row_filtered(z, 0.0, 7, 0.5, 5, row, row) == int(np.argmax(z))


def _draws(z, T, k, p, n, seed=11):
    """n draws of one row, draw i at offset i (vectorised over offsets with the oracle's own parts)."""
    V = z.shape[0]
    nb = (V + 3) // 4
    blocks = np.arange(nb, dtype=np.uint64)
    offs = np.arange(n, dtype=np.uint64)
    words = osm.philox4x32_10(blocks[None, :], 0, offs[:, None] & np.uint64(0xFFFFFFFF),
                              offs[:, None] >> np.uint64(32), seed, 0)
    w = np.stack(words, axis=2).reshape(n, nb * 4)[:, :V]
    u = ((w >> np.uint32(9)).astype(np.int64) * 2 + 1).astype(np.float32) * np.float32(2.0 ** -24)
    keys = z[None, :] * (np.float32(1.0) / np.float32(T)) + osm.gumbel_f32(u)
    keep = fl.survivors(z, T, k, p)
    masked = np.full_like(keys, -np.inf)
    masked[:, keep] = keys[:, keep]
    d = np.argmax(masked, axis=1)
    for i in [0, 1, n - 1]:
        assert d[i] == fl.sample_row_filtered(z, T, k, p, seed, i, 0)
    return d, keep


def _filtered_softmax(z, T, keep):
    q = np.zeros(z.shape[0])
    e = np.exp((z[keep].astype(np.float64) - z.max()) / T)
    q[keep] = e / e.sum()
    return q


@pytest.mark.parametrize("T,k,p", [(0.8, 10, 1.0), (1.0, 0, 0.8), (0.7, 12, 0.9)])
def test_filtered_draws_match_the_filtered_softmax_chi_squared(T, k, p):
    """20,000 draws against softmax(z / T) restricted to the survivors; nothing outside them."""
    rng = np.random.default_rng(2024)
    z = (rng.standard_normal(16) * 1.5).astype(np.float32)
    n = 20_000
    d, keep = _draws(z, T, k, p, n)
    q = _filtered_softmax(z, T, keep)
    counts = np.bincount(d, minlength=16)
    assert counts[q == 0].sum() == 0
    assert stats.chisquare(counts[keep], q[keep] * n).pvalue > 1e-3, (counts, q * n)
    # the textbook nucleus in float64 agrees where no cumulative mass lies near p
    if 0 < p < 1:
        pr = np.exp((z.astype(np.float64) - z.max()) / T)
        order = np.argsort(-z, kind="stable")
        top = order[:k] if k > 0 else order
        c = np.cumsum(pr[top]) / pr[top].sum()
        assert np.min(np.abs(c - p)) > 1e-4
        np.testing.assert_array_equal(keep, np.sort(top[:int(np.searchsorted(c, p)) + 1]))


def test_chi_squared_detects_a_missing_renormalisation():
    """Planted mistake: drawing from the unfiltered softmax after top-k fails the same check."""
    rng = np.random.default_rng(2024)
    z = (rng.standard_normal(16) * 1.5).astype(np.float32)
    n = 20_000
    d, keep = _draws(z, 0.8, 10, 1.0, n)
    q_all = _filtered_softmax(z, 0.8, np.arange(16))
    counts = np.bincount(d, minlength=16)
    assert stats.chisquare(counts, q_all * n * (counts.sum() / (q_all * n).sum())).pvalue < 1e-6
