"""Top-k / top-p filtered sampling on the GPU against the oracle, bit for bit (through the C ABI).

Both sides take every integer decision exactly (rank order, the k-th entry, the integer nucleus cut, the
float32 key of the draw), so the sampled ids and the survivor counts must agree exactly.  The rows cover
the kernel's paths: boundary buckets small enough to sort in shared memory, oversized buckets resolved by
the radix descent (all-equal rows, a bulk squeezed into one bucket by an outlier), ties, signed zeros,
greedy rows, rows with no filter, and ragged vocabularies.
"""
import numpy as np
import pytest

import oracle
from oracle import filters as fl

from harness import ensure_built

pytestmark = pytest.mark.gpu

V_FULL = 151936


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    return torch


def _run(torch, z, temps, ks, ps, seed, offset):
    from graph_replayed_decode_gb300 import eng
    rows, vocab = z.shape
    zd = torch.from_numpy(np.ascontiguousarray(z)).cuda()
    ids = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    kept = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    eng.eng_sample_filtered(zd.data_ptr(), rows, vocab, temps, ks, ps, seed, offset, ids.data_ptr(), kept.data_ptr())
    torch.cuda.synchronize()
    return ids.cpu().numpy(), kept.cpu().numpy()


def _check(torch, z, temps, ks, ps, seeds=((0, 0), (77, 2 ** 33 + 9))):
    temps = np.asarray(temps, dtype=np.float32)
    ks = np.asarray(ks, dtype=np.int32)
    ps = np.asarray(ps, dtype=np.float32)
    want_kept = oracle.survivor_counts(z, temps, ks, ps)
    for seed, offset in seeds:
        ids, kept = _run(torch, z, temps, ks, ps, seed, offset)
        want = oracle.sample_filtered(z, temps, ks, ps, seed, offset)
        np.testing.assert_array_equal(kept, want_kept)
        np.testing.assert_array_equal(ids, want)


def test_exp_f32_bit_exact(torch_cuda):
    from graph_replayed_decode_gb300 import eng
    torch = torch_cuda
    lo = int(np.array([-23.5], dtype=np.float32).view(np.uint32)[0])
    bits = np.arange(0x80000000, lo + 1, 13, dtype=np.uint64).astype(np.uint32)
    d = np.concatenate([bits.view(np.float32), np.array([0.0, -0.0, -23.0, -1e30, -np.log(2.0)], np.float32)])
    dd = torch.from_numpy(d).cuda()
    out = torch.empty_like(dd)
    eng.eng_exp_f32(dd.data_ptr(), out.data_ptr(), d.size)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), fl.exp_f32(d).view(np.uint32))


def test_filtered_sampler_bit_exact_full_vocabulary(torch_cuda):
    """Qwen vocabulary (151,936): logit spreads from flat to peaked, every filter combination."""
    rng = np.random.default_rng(21)
    rows = []
    normal3 = lambda: (rng.standard_normal(V_FULL) * 3).astype(np.float32)
    flat = lambda: (rng.standard_normal(V_FULL) * 0.5).astype(np.float32)

    def peaked():
        z = (rng.standard_normal(V_FULL) * 1.0).astype(np.float32)
        top = rng.choice(V_FULL, 30, replace=False)
        z[top] += rng.uniform(8, 14, 30).astype(np.float32)
        return z

    ties = lambda: (np.rint(rng.standard_normal(V_FULL) * 8) / 4).astype(np.float32)   # quarter steps
    cases = [
        (normal3(), 0.0, 50, 0.9),      # greedy
        (normal3(), 1.0, 0, 1.0),       # no filter
        (normal3(), 0.8, 50, 1.0),      # top-k only
        (flat(), 1.0, 0, 0.9),          # top-p only, wide nucleus
        (normal3(), 0.7, 1000, 0.95),
        (normal3(), 1.2, 20, 0.5),
        (normal3(), 1.0, 1, 0.3),
        (flat(), 1.0, V_FULL - 1, 0.999),
        (normal3(), 0.5, 0, 0.05),
        (peaked(), 1.0, 0, 0.9),
        (peaked(), 0.6, 40, 0.8),
        (ties(), 1.0, 100, 0.9),
        (ties(), 1.0, 0, 0.7),
        (ties(), 1.0, 5000, 1.0),
    ]
    z = np.stack([c[0] for c in cases])
    _check(torch_cuda, z, [c[1] for c in cases], [c[2] for c in cases], [c[3] for c in cases])


def test_oversized_boundary_buckets_take_the_radix_descent(torch_cuda):
    """All-equal rows (one bucket of 151,936 equal keys, ranked by index) and a bulk squeezed into one bucket
    by a single outlier (151,935 distinct keys in one bucket)."""
    rng = np.random.default_rng(5)
    zeros = np.zeros(V_FULL, dtype=np.float32)
    bulk = (rng.standard_normal(V_FULL) * 1e-3).astype(np.float32)
    bulk[777] = 100.0
    cases = [
        (zeros, 1.0, 100, 1.0),         # top-k by index among equal keys
        (zeros, 1.0, 0, 0.3),           # top-p: 30% of equal weights
        (zeros, 1.0, 9000, 0.5),        # both, the cut inside the top-k bucket
        (bulk, 1.0, 1000, 1.0),         # top-k inside the squeezed bulk
        (bulk, 100.0, 0, 0.6),          # top-p deep into the bulk (T = 100 flattens the outlier)
        (bulk, 100.0, 20000, 0.4),      # both inside the bulk
        (bulk, 1.0, 0, 0.5),            # the outlier alone carries the mass
    ]
    z = np.stack([c[0] for c in cases])
    _check(torch_cuda, z, [c[1] for c in cases], [c[2] for c in cases], [c[3] for c in cases])


def test_signed_zeros_and_small_ragged_vocabularies(torch_cuda):
    rng = np.random.default_rng(8)
    z = np.array([[-0.0, 0.0, -1.0, 0.0, -0.0, -2.0, -0.0]], dtype=np.float32)
    for k in [1, 2, 3, 4, 6]:
        _check(torch_cuda, z, [1.0], [k], [1.0], seeds=((3, 1),))
    for V in [1, 2, 7, 16, 4099]:
        R = 6
        zz = (rng.standard_normal((R, V)) * 2).astype(np.float32)
        temps = rng.choice([0.0, 0.7, 1.0, 1.5], R)
        ks = rng.integers(-1, V + 2, R)
        ps = rng.choice([0.0, 0.2, 0.5, 0.9, 1.0, 1.2], R)
        _check(torch_cuda, zz, temps, ks, ps)


def test_no_filter_matches_the_unfiltered_sampler(torch_cuda):
    from graph_replayed_decode_gb300 import eng
    torch = torch_cuda
    rng = np.random.default_rng(2)
    rows = 5
    z = (rng.standard_normal((rows, V_FULL)) * 3).astype(np.float32)
    temps = np.array([0.7, 1.0, 0.0, 1.3, 0.9], dtype=np.float32)
    ids, kept = _run(torch, z, temps, None, None, 4, 6)
    plain = torch.empty(rows, dtype=torch.int32, device="cuda")
    eng.eng_sample(torch.from_numpy(z).cuda().data_ptr(), rows, V_FULL, temps, 4, 6, plain.data_ptr())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids, plain.cpu().numpy())
    np.testing.assert_array_equal(kept, np.where(temps == 0, 1, V_FULL))


def test_non_finite_logits_never_survive(torch_cuda):
    rng = np.random.default_rng(4)
    z = (rng.standard_normal((3, 4096)) * 2).astype(np.float32)
    low = z.copy()
    for r, v in [(0, 5), (1, int(np.argmax(z[1]))), (2, 100)]:
        z[r, v] = [np.nan, np.inf, -np.inf][r]
        low[r, v] = -1e30                          # ranked last, never drawn, weight 0
    temps, ks, ps = [1.0, 0.8, 1.0], [50, 0, 4000], [0.9, 0.5, 1.0]
    ids, kept = _run(torch_cuda, z, np.float32(temps), np.int32(ks), np.float32(ps), 1, 2)
    np.testing.assert_array_equal(ids, oracle.sample_filtered(low, temps, ks, ps, 1, 2))
    np.testing.assert_array_equal(kept, oracle.survivor_counts(low, temps, ks, ps))


def test_filtered_sampler_rejects_bad_arguments(torch_cuda):
    from graph_replayed_decode_gb300 import eng
    torch = torch_cuda
    z = torch.zeros((2, 8), device="cuda")
    ids = torch.empty(2, dtype=torch.int32, device="cuda")
    with pytest.raises(eng.EngError):
        eng.eng_sample_filtered(z.data_ptr(), 2, 8, [1.0, -1.0], None, None, 0, 0, ids.data_ptr())
    with pytest.raises(eng.EngError):
        eng.eng_sample_filtered(z.data_ptr(), 2, 8, [1.0, 1.0], None, [0.5, float("nan")], 0, 0, ids.data_ptr())
    with pytest.raises(eng.EngError):
        eng.eng_sample_filtered(z.data_ptr(), 2, 0, [1.0, 1.0], None, None, 0, 0, ids.data_ptr())
