"""GPU sampler arithmetic against the oracle, bit for bit (through the C ABI)."""
import numpy as np
import pytest

import oracle
from oracle import sampler as osm

from harness import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    return torch


@pytest.mark.parametrize("seed,offset", [(0, 0), (0, 7), (123456789, 2 ** 33 + 5), (2 ** 63 + 11, 1)])
def test_philox_uniforms_bit_exact(torch_cuda, seed, offset):
    from graph_replayed_decode_gb300 import eng
    torch = torch_cuda
    rows, vocab = 5, 4099                                 # ragged: vocab not a multiple of 4
    out = torch.empty((rows, vocab), dtype=torch.float32, device="cuda")
    eng.eng_philox_uniforms(seed, offset, rows, vocab, out.data_ptr())
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for r in range(rows):
        np.testing.assert_array_equal(got[r].view(np.uint32), oracle.uniforms(seed, offset, r, vocab).view(np.uint32))


def test_gumbel_bit_exact_on_every_grid_uniform(torch_cuda):
    from graph_replayed_decode_gb300 import eng
    torch = torch_cuda
    k = np.arange(2 ** 23, dtype=np.int64)
    u = ((2 * k + 1).astype(np.float32)) * np.float32(2.0 ** -24)
    ud = torch.from_numpy(u).cuda()
    gd = torch.empty_like(ud)
    eng.eng_gumbel(ud.data_ptr(), gd.data_ptr(), u.size)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gd.cpu().numpy().view(np.uint32), osm.gumbel_f32(u).view(np.uint32))


def test_sampler_bit_exact_on_given_logits(torch_cuda):
    from graph_replayed_decode_gb300 import eng
    torch = torch_cuda
    rng = np.random.default_rng(3)
    rows, vocab = 7, 151936
    z = (rng.standard_normal((rows, vocab)) * 3).astype(np.float32)
    z[2, 100] = z[2, 9000] = z[2].max() + 1.0            # exact tie: lowest index wins (greedy row)
    temps = np.array([0.7, 1.0, 0.0, 0.8, 1e-3, 2.0, 0.0], dtype=np.float32)
    zd = torch.from_numpy(z).cuda()
    ids = torch.empty(rows, dtype=torch.int32, device="cuda")
    for seed, offset in [(0, 0), (99, 12345)]:
        eng.eng_sample(zd.data_ptr(), rows, vocab, temps, seed, offset, ids.data_ptr())
        torch.cuda.synchronize()
        want = oracle.sample(z, temps, seed, offset)
        np.testing.assert_array_equal(ids.cpu().numpy(), want)
    assert int(ids[2]) == 100
