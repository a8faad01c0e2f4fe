"""The fp16 variant of a model (ENG_DTYPE_F16): IEEE binary16 weights, K/V cache and operand planes, the
same kernels compiled for binary16 (the grd::f16 objects of libeng.so), against the oracle on the same
fp16 weights (widened exactly to float64).  The configuration list names "random init fp16/bf16" for the
Qwen2.5-1.5B-shaped mixed step; the tiny model covers prefill, graph-replayed decode with greedy and
Gumbel-max sampling, and the flat-partition decode attention."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from harness import GpuEngine, block_table, check_logits_and_ids
from oracle.model import widen_f16

pytestmark = pytest.mark.gpu

S = synth.shape("tiny")
NB, MBS = 64, 8


@pytest.fixture(scope="module")
def weights():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return synth.make_weights(S, seed=0, dtype="f16", norm_scale=0.1)


def _engine(w, **kw):
    args = dict(num_blocks=NB, max_reqs=8, max_tokens=128, max_blocks_per_seq=MBS)
    args.update(kw)
    return GpuEngine(S, w, **args)


@pytest.mark.parametrize("temps", [[0.0] * 4, [1.0, 0.7, 0.0, 1.3]])
def test_tiny_f16_prefill_then_graph_decode(weights, temps):
    from graph_replayed_decode_gb300.eng import StepArrays
    g = _engine(weights)
    try:
        g.capture([1, 2, 4, 8])
        pool = oracle.BlockPool(NB)
        cache = oracle.PagedCache(S, NB)
        model = oracle.OracleModel(S, weights, dtype="f16")
        R, P, steps, seed = 4, 16, 8, 5
        blocks = []
        for r in range(R):
            got = g.alloc(oracle.blocks_needed(P + steps))
            np.testing.assert_array_equal(got, pool.alloc(oracle.blocks_needed(P + steps)))
            blocks.append(list(got))
            cache.set_block_table(r, got)
        bt = block_table(blocks, MBS)
        temps = np.asarray(temps, dtype=np.float32)
        ids = np.concatenate([synth.prompt_ids(P, S.vocab, r) for r in range(R)])
        pos = np.concatenate([np.arange(P)] * R)
        cu = np.arange(R + 1) * P
        errs = []
        for k in range(steps):
            seq = np.array([pos[cu[r + 1] - 1] + 1 for r in range(R)])
            gid, glog = g.step(StepArrays(ids, pos, cu, bt, seq, temps, seed=seed, offset=k))
            assert g.info().replayed == int(k > 0)
            olog = oracle.forward_step(model, cache, ids, pos, cu)
            errs.append(check_logits_and_ids(glog, gid, olog, temps, seed, k))
            ids = gid.copy()
            pos = np.array([pos[cu[r + 1] - 1] + 1 for r in range(R)])
            cu = np.arange(R + 1)
        assert max(errs) <= 3e-2
        assert g.status() == 0
    finally:
        g.close()


def test_tiny_f16_six_rows_flat_attention(weights):
    """Six decode rows over synthetic fp16 contexts (the flat-partition decode attention), eager and then
    replayed in the bucket of 8 (bit-identical), against the oracle over the same contexts."""
    from graph_replayed_decode_gb300.eng import StepArrays
    g = _engine(weights)
    try:
        ctxs = [100, 37, 64, 17, 90, 50]
        R = len(ctxs)
        blocks = [list(g.alloc(oracle.blocks_needed(c + 1))) for c in ctxs]
        kv = {(l, r): synth.kv_context(S, l, 300 + r, c, dtype="f16") for l in range(S.layers) for r, c in enumerate(ctxs)}
        for (l, r), x in kv.items():
            g.fill_context(l, blocks[r], x)
        bt = block_table(blocks, MBS)
        ids = synth.decode_ids(R, S.vocab, 4)
        pos = np.array(ctxs)
        temps = np.zeros(R, dtype=np.float32)
        st = StepArrays(ids, pos, np.arange(R + 1), bt, pos + 1, temps)
        eid, elog = g.step(st)
        assert g.info().replayed == 0
        g.capture([8])
        rid, rlog = g.step(st)
        assert g.info().replayed == 1
        np.testing.assert_array_equal(rlog.view(np.uint32), elog.view(np.uint32))
        np.testing.assert_array_equal(rid, eid)
        model = oracle.OracleModel(S, weights, dtype="f16")
        cc = oracle.ContiguousCache(S, {r: c + 1 for r, c in enumerate(ctxs)})
        for (l, r), x in kv.items():
            cc.keys[(l, r)][:, :ctxs[r], :] = widen_f16(x[0])
            cc.values[(l, r)][:, :ctxs[r], :] = widen_f16(x[1])
        olog = oracle.forward_step(model, cc, ids, pos, np.arange(R + 1))
        assert check_logits_and_ids(elog, eid, olog, temps, 0, 0) <= 3e-2
        assert g.status() == 0
    finally:
        g.close()


def test_f16_engine_refuses_bf16_matrices(weights):
    """An fp16 engine given bf16 matrices fails at creation with ENG_EINVAL (and a message)."""
    from graph_replayed_decode_gb300 import eng
    bf = synth.make_weights(S, seed=0)
    cfg = eng.make_config(S, NB, 8, 128, MBS, dtype="f16")
    with pytest.raises(eng.EngError) as ei:
        eng.eng_create(cfg, eng.TensorList(bf.items(), "bf16"), None)
    assert ei.value.code == eng.ENG_EINVAL


def test_qwen2p5_1p5b_f16_mixed_step():
    """Qwen2.5-1.5B shape in fp16: a 512-position chunk of fresh prompts followed by 32 decode rows at
    contexts from {64, 256, 1024, 4096}, greedy, one packed step (tensor-core projections for the chunk);
    eager, then on piecewise graphs (bit-identical); logits against the oracle on the same fp16 weights."""
    from graph_replayed_decode_gb300.eng import StepArrays
    s = synth.shape("qwen2p5_1p5b")
    w = synth.make_weights(s, seed=0, dtype="f16", norm_scale=0.1)
    chunk = synth.mixed_chunk_prompts(512, key=0, seed=0)
    P = len(chunk)
    dctx = [int(c) for c in synth.context_lengths(32, (64, 256, 1024, 4096), key=1, seed=0)]
    need = [oracle.blocks_needed(plen + 1) for plen, _ in chunk] + [oracle.blocks_needed(c + 1) for c in dctx]
    mbs = max(need)
    g = GpuEngine(s, w, num_blocks=sum(need) + 4, max_reqs=64, max_tokens=600, max_blocks_per_seq=mbs)
    try:
        blocks = [list(g.alloc(n)) for n in need]
        for j, c in enumerate(dctx):
            for l in range(s.layers):
                g.fill_context(l, blocks[P + j], synth.kv_context(s, l, 100 + j, c, dtype="f16"))
        bt = block_table(blocks, mbs)
        prompts = [synth.prompt_ids(take, s.vocab, 50 + i) for i, (plen, take) in enumerate(chunk)]
        dec_ids = synth.decode_ids(32, s.vocab, 2)
        ids = np.concatenate(prompts + [dec_ids])
        pos = np.concatenate([np.arange(take) for _, take in chunk] + [np.array(dctx)])
        cu = np.concatenate([[0], np.cumsum([take for _, take in chunk] + [1] * 32)])
        seq = np.array([take for _, take in chunk] + [c + 1 for c in dctx])
        temps = np.zeros(P + 32, dtype=np.float32)
        gid, glog = g.step(StepArrays(ids, pos, cu, bt, seq, temps))
        assert g.info().num_prefill == P and g.info().replayed == 0
        g.capture_mixed([600])
        pid, plog = g.step(StepArrays(ids, pos, cu, bt, seq, temps))
        assert g.info().replayed == 2 and g.info().bucket == 600
        np.testing.assert_array_equal(pid, gid)
        np.testing.assert_array_equal(plog.view(np.uint32), glog.view(np.uint32))
        model = oracle.OracleModel(s, w, cache_layers=False, dtype="f16")
        pc = oracle.PagedCache(s, sum(need) + 4)
        for r in range(P):
            pc.set_block_table(r, blocks[r])
        t_pre = int(cu[P])
        olog = oracle.forward_step(model, pc, ids[:t_pre], pos[:t_pre], cu[:P + 1])
        check_logits_and_ids(glog, gid, olog, temps, 0, 0, rows=list(range(P)))
        rows = [P, P + int(np.argmax(dctx)), P + 31]
        cc = oracle.ContiguousCache(s, {r: dctx[r - P] + 1 for r in rows})
        for r in rows:
            for l in range(s.layers):
                kv = synth.kv_context(s, l, 100 + (r - P), dctx[r - P], dtype="f16")
                cc.keys[(l, r)][:, :dctx[r - P], :] = widen_f16(kv[0])
                cc.values[(l, r)][:, :dctx[r - P], :] = widen_f16(kv[1])
        dlog = oracle.forward_step(model, cc, ids[t_pre + np.array(rows) - P], pos[t_pre + np.array(rows) - P],
                                   np.arange(len(rows) + 1), request_keys=rows)
        check_logits_and_ids(glog, gid, dlog, temps, 0, 0, rows=rows)
        assert g.status() == 0
    finally:
        g.close()
