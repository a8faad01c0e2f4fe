"""eng_sample_noalloc: the sampler for callers that may not allocate device memory.

Some callers cannot allocate device memory while they run -- a serving runtime that has given all free
device memory to its own pool, or a latency-critical loop that cannot afford an allocation's implicit
synchronisation.  eng_sample_noalloc keeps its per-call scratch in a fixed array inside the library.  This
file checks, through the C ABI, that it returns exactly the ids of eng_sample (which allocates its scratch
per call) on two calls in a row, so the shared array's leftovers from one call cannot leak into the next,
and that it rejects more rows than its array holds.  It sits last in collection order on purpose.
"""
import numpy as np
import pytest

from harness import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    return torch


def test_noalloc_sampler_matches_eng_sample_on_two_calls(torch_cuda):
    from graph_replayed_decode_gb300 import eng
    torch = torch_cuda
    rng = np.random.default_rng(11)
    calls = [
        (9, 151936, np.array([0.7, 1.0, 0.0, 0.8, 1e-3, 2.0, 0.0, 1.3, 0.5], dtype=np.float32), 0, 0),
        (5, 4096, np.array([0.0, 1.0, 0.0, 0.9, 3.0], dtype=np.float32), 77, 123456789),
    ]
    for rows, vocab, temps, seed, offset in calls:          # two calls in a row share the fixed array
        z = torch.from_numpy((rng.standard_normal((rows, vocab)) * 3).astype(np.float32)).cuda()
        want = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
        got = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
        eng.eng_sample(z.data_ptr(), rows, vocab, temps, seed, offset, want.data_ptr())
        eng.eng_sample_noalloc(z.data_ptr(), rows, vocab, temps, seed, offset, got.data_ptr())
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.cpu().numpy(), want.cpu().numpy())
        assert (got.cpu().numpy() >= 0).all()


def test_noalloc_sampler_rejects_rows_beyond_its_array(torch_cuda):
    from graph_replayed_decode_gb300 import eng
    torch = torch_cuda
    rows, vocab = 4097, 16
    z = torch.zeros((rows, vocab), dtype=torch.float32, device="cuda")
    ids = torch.zeros(rows, dtype=torch.int32, device="cuda")
    with pytest.raises(eng.EngError) as ei:
        eng.eng_sample_noalloc(z.data_ptr(), rows, vocab, np.zeros(rows, dtype=np.float32), 0, 0, ids.data_ptr())
    assert ei.value.code == eng.ENG_EINVAL and "4096" in str(ei.value)
