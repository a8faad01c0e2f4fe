"""Pins of the oracle's sampler: Philox, the float32 log, Gumbel-max and the 20,000-draw milestone."""
import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import sampler as osm


def _triton_philox(counters: np.ndarray, seed: int) -> np.ndarray:
    """Triton's Philox4x32-10 run on its CPU interpreter (an independent library implementation)."""
    os.environ["TRITON_INTERPRET"] = "1"
    triton = pytest.importorskip("triton")
    torch = pytest.importorskip("torch")
    import triton.language as tl

    @triton.jit
    def kern(c_ptr, out_ptr, seed, N: tl.constexpr):
        i = tl.arange(0, N)
        c0 = tl.load(c_ptr + i * 4 + 0)
        c1 = tl.load(c_ptr + i * 4 + 1)
        c2 = tl.load(c_ptr + i * 4 + 2)
        c3 = tl.load(c_ptr + i * 4 + 3)
        a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
        tl.store(out_ptr + i * 4 + 0, a)
        tl.store(out_ptr + i * 4 + 1, b)
        tl.store(out_ptr + i * 4 + 2, c)
        tl.store(out_ptr + i * 4 + 3, d)

    n = counters.shape[0]
    c = torch.from_numpy(counters.astype(np.uint32).view(np.int32).copy())
    out = torch.zeros(n * 4, dtype=torch.int32)
    kern[(1,)](c, out, seed, N=n)
    return out.numpy().view(np.uint32).reshape(n, 4)


def test_philox_matches_triton_interpreter():
    rng = np.random.default_rng(5)
    counters = rng.integers(0, 2 ** 32, size=(64, 4), dtype=np.uint64).astype(np.uint32)
    counters[0] = 0
    counters[1] = 0xFFFFFFFF
    for seed in [0, 1, 0x243F6A8885A308D3 & 0x7FFFFFFFFFFFFFFF, 2 ** 40 + 17]:
        ref = _triton_philox(counters, seed)
        mine = np.stack(oracle.philox4x32_10(counters[:, 0], counters[:, 1], counters[:, 2], counters[:, 3],
                                             seed & 0xFFFFFFFF, seed >> 32), axis=1)
        np.testing.assert_array_equal(mine, ref)


def test_uniforms_open_interval_and_uniform():
    u = oracle.uniforms(seed=0, offset=3, row=5, vocab=200_000)
    assert u.dtype == np.float32 and u.min() > 0.0 and u.max() < 1.0
    assert stats.kstest(u.astype(np.float64), "uniform").pvalue > 1e-3
    lag = np.corrcoef(u[:-1].astype(np.float64), u[1:].astype(np.float64))[0, 1]
    assert abs(lag) < 0.01
    v = oracle.uniforms(seed=0, offset=4, row=5, vocab=1000)
    assert not np.array_equal(u[:1000], v)                       # a new offset draws new noise


def test_uniform_grid_values_are_exact():
    x = np.array([0, 511, 512, 0xFFFFFFFF], dtype=np.uint32)
    k = ((x >> np.uint32(9)).astype(np.int64) * 2 + 1).astype(np.float32) * np.float32(2.0 ** -24)
    np.testing.assert_array_equal(k.astype(np.float64), [2.0 ** -24, 2.0 ** -24, 3 * 2.0 ** -24,
                                                         1 - 2.0 ** -24])


def _ulp_err(a32: np.ndarray, exact: np.ndarray) -> np.ndarray:
    ulp = np.spacing(np.abs(a32).astype(np.float32)).astype(np.float64)
    return np.abs(a32.astype(np.float64) - exact) / ulp


def test_ln_f32_within_two_ulp_of_libm_on_every_grid_uniform():
    k = np.arange(2 ** 23, dtype=np.int64)
    u = ((2 * k + 1).astype(np.float32)) * np.float32(2.0 ** -24)
    lu = osm.ln_f32(u)
    err = _ulp_err(lu, np.log(u.astype(np.float64)))
    assert err.max() <= 2.0
    # second log of the Gumbel transform: arguments -ln u in [6e-8, 16.7]
    a = -lu
    err2 = _ulp_err(osm.ln_f32(a), np.log(a.astype(np.float64)))
    assert err2.max() <= 2.0


def test_ln_f32_special_points():
    x = np.array([1.0, 2.0, 0.5, 2.0 ** -24, math.e], dtype=np.float32)
    out = osm.ln_f32(x).astype(np.float64)
    np.testing.assert_allclose(out, np.log(x.astype(np.float64)), rtol=2 ** -22)
    assert out[0] == 0.0


def test_gumbel_max_with_fixed_uniforms_equals_float64_argmax():
    rng = np.random.default_rng(9)
    V, agree, checked = 4096, 0, 0
    for row in range(40):
        z = (rng.standard_normal(V) * 2.0).astype(np.float32)
        T = [0.7, 1.0, 1.3][row % 3]
        u = oracle.uniforms(17, 2, row, V)
        ours = oracle.sample_row(z, T, 17, 2, row)
        key64 = z.astype(np.float64) / T - np.log(-np.log(u.astype(np.float64)))
        srt = np.sort(key64)
        if srt[-1] - srt[-2] > 1e-5:
            checked += 1
            agree += int(ours == int(np.argmax(key64)))
    assert checked >= 35 and agree == checked


def test_greedy_and_tie_break():
    z = np.array([0.5, 2.0, -1.0, 2.0], dtype=np.float32)
    assert oracle.sample_row(z, 0.0, 0, 0, 0) == 1                        # ties go to the lowest index
    z2 = np.array([0.1, 3.0, 2.9, -5.0], dtype=np.float32)
    draws = [oracle.sample_row(z2, 1e-4, 0, off, 0) for off in range(50)]  # T -> 0 is the argmax
    assert set(draws) == {1}


@pytest.mark.parametrize("temperature", [0.7, 1.0])
def test_gumbel_max_frequencies_match_softmax_chi_squared(temperature):
    """The milestone of "19. Fast decode": 20,000 draws against softmax(z / T), 16-way vocabulary."""
    rng = np.random.default_rng(2024)
    z = (rng.standard_normal(16) * 1.5).astype(np.float32)
    n = 20_000
    # draw n samples: each draw is one (offset) of the same row
    blocks = np.arange(4, dtype=np.uint64)
    offs = np.arange(n, dtype=np.uint64)
    words = osm.philox4x32_10(blocks[None, :], 0, offs[:, None] & np.uint64(0xFFFFFFFF), offs[:, None] >> np.uint64(32),
                              11, 0)
    w = np.stack(words, axis=2).reshape(n, 16)
    u = ((w >> np.uint32(9)).astype(np.int64) * 2 + 1).astype(np.float32) * np.float32(2.0 ** -24)
    inv_t = np.float32(1.0) / np.float32(temperature)
    keys = z[None, :] * inv_t + osm.gumbel_f32(u)
    draws = np.argmax(keys, axis=1)
    # the vectorised draws are the sampler's own draws
    for i in [0, 1, 777, n - 1]:
        assert draws[i] == oracle.sample_row(z, temperature, 11, i, 0)
    p = np.exp(z.astype(np.float64) / temperature)
    p /= p.sum()
    counts = np.bincount(draws, minlength=16)
    chi = stats.chisquare(counts, p * n)
    assert chi.pvalue > 1e-3, (counts, p * n)


def test_chi_squared_detects_missing_temperature():
    """Planted mistake: ignoring the temperature must fail the same chi-squared check."""
    rng = np.random.default_rng(2024)
    z = (rng.standard_normal(16) * 1.5).astype(np.float32)
    n = 20_000
    blocks = np.arange(4, dtype=np.uint64)
    offs = np.arange(n, dtype=np.uint64)
    words = osm.philox4x32_10(blocks[None, :], 0, offs[:, None], 0, 11, 0)
    w = np.stack(words, axis=2).reshape(n, 16)
    u = ((w >> np.uint32(9)).astype(np.int64) * 2 + 1).astype(np.float32) * np.float32(2.0 ** -24)
    draws = np.argmax(z[None, :] + osm.gumbel_f32(u), axis=1)             # T = 0.7 forgotten
    p = np.exp(z.astype(np.float64) / 0.7)
    p /= p.sum()
    assert stats.chisquare(np.bincount(draws, minlength=16), p * n).pvalue < 1e-6
