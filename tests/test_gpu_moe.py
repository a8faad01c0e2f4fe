"""The mixture-of-experts calls ("33. Removing overhead", §A MoE layer that never asks the host) against the
oracle (oracle/moe.py): the grouping bit for bit, the router's experts and weights, the grouped layer against
the per-token definition on a small ragged case and on the Qwen3-30B-A3B-shaped layer, and a CUDA-graph replay
with a different routing written into the same buffers (no shape depends on the routing)."""
from __future__ import annotations

import numpy as np
import pytest

import synth
from oracle import moe
from oracle.model import widen_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from graph_replayed_decode_gb300 import eng
    eng.lib()
    return torch


def _dev(torch, a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def _align(torch, ids, E, bm):
    from graph_replayed_decode_gb300 import eng
    N, k = ids.shape
    M = eng.eng_moe_padded_rows(N, k, E, bm)
    d_ids = _dev(torch, ids.astype(np.int32))
    s = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    b = torch.full((M // bm,), -7, dtype=torch.int32, device="cuda")
    info = torch.zeros(2, dtype=torch.int32, device="cuda")
    eng.eng_moe_align(d_ids.data_ptr(), N, k, E, bm, s.data_ptr(), b.data_ptr(), info.data_ptr())
    torch.cuda.synchronize()
    return s.cpu().numpy(), b.cpu().numpy(), info.cpu().numpy()


@pytest.mark.parametrize("N,k,E,bm", [(1, 1, 1, 16), (7, 2, 8, 16), (40, 8, 128, 16), (33, 2, 4, 64), (5, 8, 16, 4),
                                      (512, 8, 128, 16), (2000, 8, 128, 16), (64, 8, 128, 64)])
def test_align_matches_the_oracle_bit_for_bit(cuda, N, k, E, bm):
    rng = np.random.default_rng(N * 7 + E)
    for trial in range(3):
        if trial == 0:
            ids = np.full((N, k), E - 1, dtype=np.int64)             # every assignment on the last expert
        else:
            ids = np.stack([rng.choice(E, size=k, replace=k > E) for _ in range(N)])
        s, b, info = _align(cuda, ids, E, bm)
        want_s, want_b, want_n = moe.moe_align(ids, E, bm)
        np.testing.assert_array_equal(s, want_s)
        np.testing.assert_array_equal(b, want_b)
        assert info[0] == want_n and info[1] == 0


def test_align_reports_out_of_range_ids(cuda):
    ids = np.array([[0, 3], [9, 1], [2, -1]], dtype=np.int64)          # 9 and -1 are outside [0, 4)
    s, b, info = _align(cuda, ids, 4, 2)
    assert info[1] == 2
    placed = sorted(int(v) for v in s if v < ids.size)
    assert placed == [0, 1, 3, 4]                                     # the in-range assignments, once each


@pytest.mark.parametrize("name,N", [("tiny_moe", 19), ("qwen3_30b_a3b_moe", 48)])
def test_router_matches_the_oracle(cuda, name, N):
    torch = cuda
    from graph_replayed_decode_gb300 import eng
    m = synth.moe_shape(name)
    w = synth.moe_weights(m, seed=0)
    x = synth.moe_tokens(N, m.hidden, key=1)
    wts = torch.zeros((N, m.top_k), dtype=torch.float32, device="cuda")
    ids = torch.zeros((N, m.top_k), dtype=torch.int32, device="cuda")
    dx, dr = _dev(torch, x), _dev(torch, w["router"])      # held: the calls take raw device pointers
    eng.eng_moe_route(dx.data_ptr(), dr.data_ptr(), N, m.hidden, m.experts, m.top_k, wts.data_ptr(), ids.data_ptr())
    torch.cuda.synchronize()
    gw, gi = wts.cpu().numpy(), ids.cpu().numpy()
    ow, oi = moe.route(widen_bf16(x), widen_bf16(w["router"]), m.top_k)
    # the experts where the ranking is decided by more than float32 rounding of the logits
    logits = widen_bf16(x) @ widen_bf16(w["router"]).T
    srt = -np.sort(-logits, axis=1)
    clear = np.min(np.abs(np.diff(srt[:, :m.top_k + 1], axis=1)), axis=1) > 1e-4
    assert clear.mean() > 0.8
    np.testing.assert_array_equal(gi[clear], oi[clear])
    np.testing.assert_allclose(gw[clear], ow[clear], rtol=1e-4, atol=1e-6)
    np.testing.assert_allclose(gw.sum(axis=1), 1.0, atol=1e-5)


def _run_mlp(torch, m, x, w, rw, ids):
    from graph_replayed_decode_gb300 import eng
    N = x.shape[0]
    out = torch.full((N, m.hidden), np.nan, dtype=torch.float32, device="cuda")
    nbytes = eng.eng_moe_workspace_bytes(N, m.top_k, m.experts, m.hidden, m.intermediate)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d = dict(x=_dev(torch, x), gu=_dev(torch, w["gate_up"]), dn=_dev(torch, w["down"]),
             rw=_dev(torch, rw.astype(np.float32)), ids=_dev(torch, ids.astype(np.int32)))
    eng.eng_moe_mlp(d["x"].data_ptr(), d["gu"].data_ptr(), d["dn"].data_ptr(), d["rw"].data_ptr(), d["ids"].data_ptr(),
                    N, m.hidden, m.intermediate, m.experts, m.top_k, out.data_ptr(), ws.data_ptr(), nbytes)
    torch.cuda.synchronize()
    return out.cpu().numpy(), d, ws, out


def _routing(m, x, w):
    return moe.route(widen_bf16(x), widen_bf16(w["router"]), m.top_k)


@pytest.mark.parametrize("name,N", [("small", 37), ("qwen3_30b_a3b_moe", 64)])
def test_grouped_layer_matches_the_per_token_definition(cuda, name, N):
    torch = cuda
    m = (synth.MoeShape("small_moe", hidden=128, experts=8, top_k=2, intermediate=64) if name == "small"
         else synth.moe_shape(name))
    w = synth.moe_weights(m, seed=0)
    x = synth.moe_tokens(N, m.hidden, key=2)
    rw, ids = _routing(m, x, w)
    got, *_ = _run_mlp(torch, m, x, w, rw, ids)
    want = moe.moe_reference(widen_bf16(x), widen_bf16(w["gate_up"]), widen_bf16(w["down"]), rw, ids)
    scale = np.abs(want).max()
    assert np.isfinite(got).all()
    # bf16 weights and inputs exact; the activation carried as a bf16 hi/lo pair; float32 accumulation
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-4 * scale)


def test_graph_replay_with_a_new_routing(cuda):
    """The layer captured once in a CUDA graph; a different routing written into the same id and weight
    buffers is replayed and matches the eager call on that routing (no launch shape depends on it)."""
    torch = cuda
    from graph_replayed_decode_gb300 import eng
    m = synth.MoeShape("small_moe", hidden=128, experts=8, top_k=2, intermediate=64)
    w = synth.moe_weights(m, seed=0)
    N = 24
    x = synth.moe_tokens(N, m.hidden, key=3)
    rw, ids = _routing(m, x, w)
    first, d, ws, out = _run_mlp(torch, m, x, w, rw, ids)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        eng.eng_moe_mlp(d["x"].data_ptr(), d["gu"].data_ptr(), d["dn"].data_ptr(), d["rw"].data_ptr(),
                        d["ids"].data_ptr(), N, m.hidden, m.intermediate, m.experts, m.top_k, out.data_ptr(),
                        ws.data_ptr(), ws.numel(), stream.cuda_stream)
    rng = np.random.default_rng(5)
    ids2 = np.stack([rng.choice(m.experts, size=m.top_k, replace=False) for _ in range(N)])
    ids2[:8] = [0, 1]                                                  # a crowded pair of experts
    rw2 = rng.random((N, m.top_k))
    rw2 /= rw2.sum(axis=1, keepdims=True)
    d["ids"].copy_(torch.from_numpy(ids2.astype(np.int32)))
    d["rw"].copy_(torch.from_numpy(rw2.astype(np.float32)))
    out.fill_(np.nan)
    graph.replay()
    torch.cuda.synchronize()
    replayed = out.cpu().numpy()
    eager, *_ = _run_mlp(torch, m, x, w, rw2, ids2)
    np.testing.assert_array_equal(replayed, eager)
    assert not np.array_equal(replayed, first)
