"""End-to-end parity on the tiny two-layer decoder: one packed prefill step then graph-replayed decode.

Workload: 4 requests with 16-token uniform-random prompts, block size 16, one packed prefill step followed
by 15 pure-decode steps (16 sampled tokens per request), greedy; and the same with Gumbel-max sampling.
Both sides consume the GPU's sampled ids (teacher forcing).

The weights' RMSNorm and QK-norm vectors are bf16 draws of 1 + N(0, 0.1^2), different for every norm and
layer, so that each norm-weight multiply fused into a projection's prologue or epilogue is checked (and the
order of QK-norm and RoPE, which unit weights cannot tell apart); one case keeps the unit weights of the
benchmark's recipe.
"""
import numpy as np
import pytest

import oracle
import synth

from harness import GpuEngine, block_table, check_logits_and_ids

pytestmark = pytest.mark.gpu

S = synth.shape("tiny")
NB, MBS = 64, 8


@pytest.fixture(scope="module")
def weights():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return synth.make_weights(S, seed=0, norm_scale=0.1)


@pytest.fixture(scope="module")
def unit_norm_weights():
    return synth.make_weights(S, seed=0)


def _engine(weights, stream=None, decode_kernel=True, num_blocks=NB, mbs=MBS):
    """An engine over the tiny shape.  decode_kernel=False keeps small decode-only steps on the per-layer
    kernels (ENG_DECODE_KERNEL=0 when the engine is created) instead of the persistent decode kernel."""
    import os
    old = os.environ.get("ENG_DECODE_KERNEL")
    os.environ["ENG_DECODE_KERNEL"] = "1" if decode_kernel else "0"
    try:
        return GpuEngine(S, weights, num_blocks=num_blocks, max_reqs=8, max_tokens=128, max_blocks_per_seq=mbs,
                         stream=stream)
    finally:
        if old is None:
            del os.environ["ENG_DECODE_KERNEL"]
        else:
            os.environ["ENG_DECODE_KERNEL"] = old


def run_tiny(weights, temps, capture=True, steps=16, seed=5):
    g = _engine(weights)
    try:
        if capture:
            g.capture([1, 2, 4, 8])
        pool = oracle.BlockPool(NB)
        cache = oracle.PagedCache(S, NB)
        model = oracle.OracleModel(S, weights)
        R, P = 4, 16
        prompts = [synth.prompt_ids(P, S.vocab, r) for r in range(R)]
        blocks = []
        for r in range(R):
            got = g.alloc(oracle.blocks_needed(P + steps))
            want = pool.alloc(oracle.blocks_needed(P + steps))
            np.testing.assert_array_equal(got, want)                 # block tables bit-exact
            blocks.append(list(got))
            cache.set_block_table(r, got)
        bt = block_table(blocks, MBS)
        temps = np.asarray(temps, dtype=np.float32)

        from graph_replayed_decode_gb300.eng import StepArrays
        ids = np.concatenate(prompts)
        pos = np.concatenate([np.arange(P)] * R)
        cu = np.arange(R + 1) * P
        errs = []
        for k in range(steps):
            seq = np.array([pos[cu[r + 1] - 1] + 1 for r in range(R)])
            st = StepArrays(ids, pos, cu, bt, seq, temps, seed=seed, offset=k)
            gid, glog = g.step(st)
            info = g.info()
            assert info.replayed == int(capture and k > 0)
            olog = oracle.forward_step(model, cache, ids, pos, cu)
            errs.append(check_logits_and_ids(glog, gid, olog, temps, seed, k))
            # slots of this step: bit-exact against the oracle's slot mapping
            import torch
            sp, _ = g.eng.eng_debug_buffer(g.h, "slots")
            from harness import device_view
            slots = device_view(sp, 4 * len(ids), torch.int32).cpu().numpy()
            want_slots = [cache.slot(int(np.searchsorted(cu, t, side="right") - 1), int(pos[t])) for t in range(len(ids))]
            np.testing.assert_array_equal(slots, want_slots)
            ids = gid.copy()
            pos = np.array([pos[cu[r + 1] - 1] + 1 for r in range(R)])
            cu = np.arange(R + 1)
        assert g.status() == 0
        return errs
    finally:
        g.close()


def test_tiny_greedy_prefill_then_graph_decode(weights):
    errs = run_tiny(weights, [0.0] * 4)
    assert max(errs) <= 3e-2


def test_tiny_greedy_unit_norm_weights(unit_norm_weights):
    errs = run_tiny(unit_norm_weights, [0.0] * 4, steps=6)
    assert max(errs) <= 3e-2


def test_tiny_gumbel_prefill_then_graph_decode(weights):
    errs = run_tiny(weights, [1.0, 0.7, 0.0, 1.3])
    assert max(errs) <= 3e-2


def test_tiny_eager_only(weights):
    run_tiny(weights, [0.0, 1.0, 0.0, 0.5], capture=False, steps=4)


def _decode_batch(g, weights, R, ctx=37, seed=0):
    """R decode rows over synthetic contexts; returns StepArrays."""
    from graph_replayed_decode_gb300.eng import StepArrays
    blocks = []
    for r in range(R):
        b = g.alloc(oracle.blocks_needed(ctx + 1))
        blocks.append(list(b))
        for l in range(S.layers):
            g.fill_context(l, b, synth.kv_context(S, l, r, ctx))
    bt = block_table(blocks, MBS)
    ids = synth.decode_ids(R, S.vocab, 0)
    pos = np.full(R, ctx)
    return StepArrays(ids, pos, np.arange(R + 1), bt, pos + 1, np.array([0.0, 1.0, 0.7, 0.0, 2.0][:R] * 2)[:R],
                      seed=seed, offset=3)


def test_graph_replay_equals_eager_bit_exact_and_padding_is_harmless(weights):
    g = _engine(weights)
    try:
        st = _decode_batch(g, weights, 3)
        ids_e, log_e = g.step(st)                        # eager (nothing captured yet)
        assert g.info().replayed == 0
        g.capture([4, 8])
        ids_g, log_g = g.step(st)                        # replayed in bucket 4 with one padding row
        info = g.info()
        assert info.replayed == 1 and info.bucket == 4
        np.testing.assert_array_equal(ids_g, ids_e)
        np.testing.assert_array_equal(log_g.view(np.uint32), log_e.view(np.uint32))
        assert np.isfinite(log_g).all()
        assert g.status() == 0
    finally:
        g.close()


def test_capture_writes_only_the_scratch_block(weights):
    import torch
    g = _engine(weights)
    try:
        _decode_batch(g, weights, 2)
        before = g.kv_pool().clone()
        g.capture([1, 2, 4, 8])
        after = g.kv_pool()
        torch.cuda.synchronize()
        assert torch.equal(before[:, :, :NB], after[:, :, :NB])
    finally:
        g.close()


def test_freed_block_poisoning_leaves_outputs_unchanged(weights):
    import torch
    g = _engine(weights)
    try:
        g.capture([4])
        st = _decode_batch(g, weights, 3, ctx=29)
        ids0, log0 = g.step(st)
        used = set(int(b) for b in st.block_tables.reshape(-1) if b)
        used |= {int(st.block_tables[0, 0])}
        pool = g.kv_pool()
        nan_bits = 0x7FC0
        free = [b for b in range(NB + 1) if b not in used]
        pool[:, :, torch.as_tensor(free, device="cuda")] = nan_bits
        # poison the tails of the last blocks too (positions past each row's length)
        for r in range(3):
            last = int(st.block_tables[r, (29 + 1 - 1) // 16])
            pool[:, :, last, :, (30 % 16):, :] = nan_bits
        ids1, log1 = g.step(st)
        np.testing.assert_array_equal(ids1, ids0)
        np.testing.assert_array_equal(log1.view(np.uint32), log0.view(np.uint32))
    finally:
        g.close()


def test_mixed_step_prefill_chunks_and_decode_rows(weights):
    """A packed step with two prompt chunks (one resuming after an earlier chunk) and three decode rows."""
    from graph_replayed_decode_gb300.eng import StepArrays
    g = _engine(weights)
    try:
        model = oracle.OracleModel(S, weights)
        cache = oracle.PagedCache(S, NB)
        blocks = [list(g.alloc(n)) for n in (3, 2, 2, 2, 3)]
        for r, b in enumerate(blocks):
            cache.set_block_table(r, b)
        bt = block_table(blocks, MBS)
        # request 0: first chunk of 20 prompt tokens, then a second chunk of 9 (positions 20..28)
        p0 = synth.prompt_ids(29, S.vocab, 10)
        first = StepArrays(p0[:20], np.arange(20), [0, 20], bt[:1], [20], [0.0])
        gid, glog = g.step(first)
        olog = oracle.forward_step(model, cache, p0[:20], np.arange(20), [0, 20])
        check_logits_and_ids(glog, gid, olog, [0.0], 0, 0)
        # decode rows 2..4 with synthetic contexts of 17, 5, 31 keys
        ctxs = [17, 5, 31]
        for j, ctx in enumerate(ctxs):
            r = 2 + j
            for l in range(S.layers):
                kv = synth.kv_context(S, l, 100 + r, ctx)
                g.fill_context(l, blocks[r], kv)
                from oracle.model import widen_bf16
                K = np.swapaxes(widen_bf16(kv[0]), 0, 1)
                V = np.swapaxes(widen_bf16(kv[1]), 0, 1)
                cache.write(l, r, np.arange(ctx), K, V)
        p1 = synth.prompt_ids(11, S.vocab, 11)
        dec = synth.decode_ids(3, S.vocab, 4)
        ids = np.concatenate([p0[20:], p1, dec])
        pos = np.concatenate([np.arange(20, 29), np.arange(11), np.array(ctxs)])
        cu = np.array([0, 9, 20, 21, 22, 23])
        seq = np.array([29, 11, 18, 6, 32])
        temps = np.array([0.0, 0.9, 0.0, 1.0, 0.0], dtype=np.float32)
        st = StepArrays(ids, pos, cu, bt, seq, temps, seed=1, offset=2)
        gid, glog = g.step(st)
        assert g.info().num_prefill == 2
        olog = oracle.forward_step(model, cache, ids, pos, cu)
        check_logits_and_ids(glog, gid, olog, temps, 1, 2)
        assert g.status() == 0
    finally:
        g.close()


def test_piecewise_graphs_for_a_mixed_step(weights):
    """eng_capture_mixed ("(7) Graph Mode", §PIECEWISE): a mixed step of 78 tokens (prompt chunks of 40 and
    35 and three decode rows) replays the 128-token projection pieces with attention launched between them.
    Ids, logits and KV slots equal the eager step's bit for bit, the next decode step agrees too (the pieces
    wrote the same K/V, the padding tokens only the scratch block), and the logits match the oracle."""
    import torch
    from graph_replayed_decode_gb300.eng import StepArrays
    from harness import device_view
    pw, eg = _engine(weights), _engine(weights)
    try:
        pw.capture_mixed([128])
        model = oracle.OracleModel(S, weights)
        cache = oracle.PagedCache(S, NB)
        ctxs = [17, 5, 31]
        blocks = None
        for g in (pw, eg):
            b = [list(g.alloc(n)) for n in (3, 3, 2, 2, 3)]
            assert blocks is None or b == blocks
            blocks = b
            for j, ctx in enumerate(ctxs):
                for l in range(S.layers):
                    g.fill_context(l, blocks[2 + j], synth.kv_context(S, l, 100 + j, ctx))
        for r, b in enumerate(blocks):
            cache.set_block_table(r, b)
        for j, ctx in enumerate(ctxs):
            for l in range(S.layers):
                kv = synth.kv_context(S, l, 100 + j, ctx)
                K = np.swapaxes(oracle.widen_bf16(kv[0]), 0, 1)
                V = np.swapaxes(oracle.widen_bf16(kv[1]), 0, 1)
                cache.write(l, 2 + j, np.arange(ctx), K, V)
        bt = block_table(blocks, MBS)
        ids = np.concatenate([synth.prompt_ids(40, S.vocab, 70), synth.prompt_ids(35, S.vocab, 71),
                              synth.decode_ids(3, S.vocab, 6)])
        pos = np.concatenate([np.arange(40), np.arange(35), np.array(ctxs)])
        cu = np.array([0, 40, 75, 76, 77, 78])
        seq = np.array([40, 35, 18, 6, 32])
        temps = np.array([0.0, 0.8, 0.0, 1.1, 0.0], dtype=np.float32)
        st = StepArrays(ids, pos, cu, bt, seq, temps, seed=4, offset=1)
        pid, plog = pw.step(st)
        info = pw.info()
        assert info.replayed == 2 and info.bucket == 128 and info.num_prefill == 2
        eid, elog = eg.step(st)
        assert eg.info().replayed == 0 and info.launches == eg.info().launches   # the same kernels
        np.testing.assert_array_equal(pid, eid)
        np.testing.assert_array_equal(plog.view(np.uint32), elog.view(np.uint32))
        slots = []
        for g in (pw, eg):
            sp, _ = g.eng.eng_debug_buffer(g.h, "slots")
            slots.append(device_view(sp, 4 * len(ids), torch.int32).cpu().numpy())
        np.testing.assert_array_equal(slots[0], slots[1])
        olog = oracle.forward_step(model, cache, ids, pos, cu)
        check_logits_and_ids(plog, pid, olog, temps, 4, 1)
        # one decode step of every request, on the K/V each engine wrote
        nxt = StepArrays(pid, seq, np.arange(6), bt, seq + 1, temps, seed=4, offset=2)
        a_ids, a_log = pw.step(nxt)
        b_ids, b_log = eg.step(nxt)
        np.testing.assert_array_equal(a_ids, b_ids)
        np.testing.assert_array_equal(a_log.view(np.uint32), b_log.view(np.uint32))
        assert pw.status() == 0 and eg.status() == 0
    finally:
        pw.close()
        eg.close()


def test_step_does_not_wait_for_the_gpu(weights):
    """eng_step returns while earlier work on its stream is still running (no host sync in the step)."""
    import torch
    from graph_replayed_decode_gb300 import eng
    stream = torch.cuda.Stream()
    g = _engine(weights, stream=stream)
    try:
        g.capture([4])
        st = _decode_batch(g, weights, 4)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(200_000_000)               # keep the stream busy for a while
        eng.eng_step(g.h, st, g.ids_dev.data_ptr(), None)
        assert not stream.query(), "eng_step waited for the stream"
        stream.synchronize()
    finally:
        g.close()


def test_host_validation_errors(weights):
    from graph_replayed_decode_gb300 import eng
    from graph_replayed_decode_gb300.eng import StepArrays
    g = _engine(weights)
    try:
        b = list(g.alloc(2))
        bt = block_table([b, b], MBS)
        with pytest.raises(eng.EngError) as ei:    # decode row before a prefill chunk
            g.step(StepArrays([1, 2, 3], [5, 0, 1], [0, 1, 3], bt, [6, 2], [0, 0]))
        assert ei.value.code == eng.ENG_EINVAL
        with pytest.raises(eng.EngError) as ei:    # position past the capacity
            bt_wide = np.zeros((1, MBS), dtype=np.int32)
            g.step(StepArrays([1], [MBS * 16], [0, 1], bt_wide, [MBS * 16 + 1], [0]))
        assert ei.value.code == eng.ENG_ECAPACITY
        with pytest.raises(eng.EngError) as ei:    # block id out of range
            g.step(StepArrays([1], [3], [0, 1], np.array([[NB + 5]]), [4], [0]))
        assert ei.value.code == eng.ENG_EINVAL
        with pytest.raises(eng.EngError) as ei:    # pool exhaustion
            g.alloc(NB)
        assert ei.value.code == eng.ENG_EPOOL
        with pytest.raises(eng.EngError):
            eng.eng_pool_free(g.h, [NB - 1])
        assert g.status() == 0
    finally:
        g.close()


def test_device_decode_loop_equals_host_driven_steps(weights):
    """eng_decode (sampled ids fed back on the device) == eng_step with the ids read back each step."""
    import torch
    from graph_replayed_decode_gb300 import eng
    from graph_replayed_decode_gb300.eng import StepArrays
    g = _engine(weights)
    try:
        g.capture([4, 8])
        st = _decode_batch(g, weights, 3, ctx=20)
        ids0, _ = g.step(st)
        n = 6
        ring = torch.zeros((n, 3), dtype=torch.int32, device="cuda")
        eng.eng_decode(g.h, n, ring.data_ptr())
        torch.cuda.synchronize()
        assert g.info().replayed == 1
        dev = np.concatenate([ids0[None], ring.cpu().numpy()])
        ids, pos = st.token_ids.copy(), st.positions.copy()
        host = []
        for k in range(n + 1):
            s2 = StepArrays(ids, pos, np.arange(4), st.block_tables, pos + 1, st.temperature, seed=st.step.seed,
                            offset=st.step.offset + k)
            ids, _ = g.step(s2, want_logits=False)
            host.append(ids.copy())
            pos = pos + 1
        np.testing.assert_array_equal(dev, np.stack(host))
        prof = eng.eng_profile(g.h)
        kinds = [k for k, _, _ in prof]
        assert kinds == ["decode_layers", "lm_head", "advance"]   # the persistent kernel runs every layer
        assert all(ms > 0 for _, ms, _ in prof)
        with pytest.raises(eng.EngError) as ei:          # past the block tables' capacity
            eng.eng_decode(g.h, 200, ring.data_ptr())
        assert ei.value.code == eng.ENG_ECAPACITY
        assert g.status() == 0
    finally:
        g.close()


def test_attention_launch_shapes_agree(weights):
    """Decode rows on the two decode-attention launch shapes -- splits merged on chip (a batch of 4 rows)
    and the flat partition over every row's blocks (the same rows plus two more) -- agree to float32
    rounding, and the flat partition gives the same bits when the step is repeated (its split points
    depend only on the step's lengths).  (Per-layer kernels: small decode steps otherwise run on the
    persistent decode kernel.)"""
    from graph_replayed_decode_gb300.eng import StepArrays
    g = _engine(weights, decode_kernel=False)
    try:
        ctxs = [100, 37, 64, 17, 90, 50]                      # 2..7 blocks: segments split between warps
        blocks = [list(g.alloc(oracle.blocks_needed(c + 1))) for c in ctxs]
        for l in range(S.layers):
            for r, c in enumerate(ctxs):
                g.fill_context(l, blocks[r], synth.kv_context(S, l, 200 + r, c))
        bt = block_table(blocks, MBS)
        ids = synth.decode_ids(6, S.vocab, 9)
        pos = np.array(ctxs)
        temps = np.zeros(6, dtype=np.float32)
        a_ids, a_log = g.step(StepArrays(ids[:4], pos[:4], np.arange(5), bt[:4], pos[:4] + 1, temps[:4]))
        b_ids, b_log = g.step(StepArrays(ids, pos, np.arange(7), bt, pos + 1, temps))
        c_ids, c_log = g.step(StepArrays(ids, pos, np.arange(7), bt, pos + 1, temps))
        np.testing.assert_array_equal(b_log.view(np.uint32), c_log.view(np.uint32))
        np.testing.assert_array_equal(b_ids, c_ids)
        np.testing.assert_allclose(b_log[:4], a_log, rtol=0, atol=2e-4)
        top2 = -np.sort(-a_log, axis=1)[:, :2]
        clear = top2[:, 0] - top2[:, 1] > 1e-3
        np.testing.assert_array_equal(a_ids[clear], b_ids[:4][clear])
        assert g.status() == 0
    finally:
        g.close()


def test_persistent_decode_kernel_matches_oracle_and_per_layer_kernels(weights):
    """The persistent decode kernel (every layer of a decode step of up to 8 tokens in one launch) against
    the oracle, on rows whose contexts span up to five attention splits (so the split merge runs) and a
    row of one block; the per-layer kernels on the same inputs land within the same bar.  Eager (3 rows)
    and replayed (bucket 4, one padding row) steps agree bit for bit, and the device loop continues them."""
    import torch
    from graph_replayed_decode_gb300 import eng
    from graph_replayed_decode_gb300.eng import StepArrays
    mbs, nb = 48, 160
    ctxs = [600, 37, 250]
    engines = [_engine(weights, decode_kernel=k, num_blocks=nb, mbs=mbs) for k in (True, False)]
    try:
        blocks = None
        for g in engines:
            b = [list(g.alloc(oracle.blocks_needed(c + 4))) for c in ctxs]
            assert blocks is None or b == blocks
            blocks = b
            for l in range(S.layers):
                for r, c in enumerate(ctxs):
                    g.fill_context(l, blocks[r], synth.kv_context(S, l, 300 + r, c))
        bt = block_table(blocks, mbs)
        model = oracle.OracleModel(S, weights)
        cache = oracle.ContiguousCache(S, {r: c + 4 for r, c in enumerate(ctxs)})
        for l in range(S.layers):
            for r, c in enumerate(ctxs):
                kv = synth.kv_context(S, l, 300 + r, c)
                cache.keys[(l, r)][:, :c, :] = oracle.widen_bf16(kv[0])
                cache.values[(l, r)][:, :c, :] = oracle.widen_bf16(kv[1])
        ids = synth.decode_ids(3, S.vocab, 5)
        pos = np.array(ctxs)
        temps = np.array([0.0, 0.9, 1.3], dtype=np.float32)
        st = StepArrays(ids, pos, np.arange(4), bt, pos + 1, temps, seed=2, offset=0)
        fast, slow = engines
        f_ids, f_log = fast.step(st)                               # eager, persistent kernel
        assert fast.info().launches == 3                           # the kernel, the LM head, the advance
        s_ids, s_log = slow.step(st)                               # eager, per-layer kernels
        assert slow.info().launches > 2 * S.layers
        olog = oracle.forward_step(model, cache, ids, pos, np.arange(4))
        check_logits_and_ids(f_log, f_ids, olog, temps, 2, 0)
        check_logits_and_ids(s_log, s_ids, olog, temps, 2, 0)
        # the same step replayed in bucket 4 (one padding row) is bit-identical to the eager one
        for g in engines:
            g.capture([4, 8])
        r_ids, r_log = fast.step(st)
        assert fast.info().replayed == 1 and fast.info().bucket == 4
        np.testing.assert_array_equal(r_ids, f_ids)
        np.testing.assert_array_equal(r_log.view(np.uint32), f_log.view(np.uint32))
        # two more steps on the device, checked against the oracle
        ring = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
        eng.eng_decode(fast.h, 2, ring.data_ptr())
        torch.cuda.synchronize()
        cur, p = f_ids.copy(), pos + 1
        for k in range(2):
            z = oracle.forward_step(model, cache, cur, p, np.arange(4))
            want = oracle.sample(z.astype(np.float32), temps, 2, k + 1)
            got = ring[k].cpu().numpy()
            for r in range(3):
                srt = np.sort(z[r])
                if temps[r] == 0.0 and srt[-1] - srt[-2] > 0.1:
                    assert got[r] == want[r]
            cur, p = got.copy(), p + 1
        assert fast.status() == 0 and slow.status() == 0
    finally:
        for g in engines:
            g.close()


def test_tensor_core_prefill_chunks(weights):
    """A packed prefill step of 127 tokens (two prompts of 70 and 57; two 64-token chunks, the second
    ragged) runs its projections on the tcgen05 path; logits and slots match the oracle."""
    from graph_replayed_decode_gb300.eng import StepArrays
    import torch
    from harness import device_view
    g = _engine(weights)
    try:
        model = oracle.OracleModel(S, weights)
        cache = oracle.PagedCache(S, NB)
        lens = [70, 57]
        blocks = [list(g.alloc(oracle.blocks_needed(n))) for n in lens]
        for r, b in enumerate(blocks):
            cache.set_block_table(r, b)
        bt = block_table(blocks, MBS)
        ids = np.concatenate([synth.prompt_ids(n, S.vocab, 40 + r) for r, n in enumerate(lens)])
        pos = np.concatenate([np.arange(n) for n in lens])
        cu = np.array([0, 70, 127])
        temps = np.array([0.0, 0.9], dtype=np.float32)
        gid, glog = g.step(StepArrays(ids, pos, cu, bt, np.array(lens), temps, seed=2, offset=0))
        assert g.info().num_prefill == 2
        olog = oracle.forward_step(model, cache, ids, pos, cu)
        check_logits_and_ids(glog, gid, olog, temps, 2, 0)
        sp, _ = g.eng.eng_debug_buffer(g.h, "slots")
        slots = device_view(sp, 4 * len(ids), torch.int32).cpu().numpy()
        want = [cache.slot(int(np.searchsorted(cu, t, side="right") - 1), int(pos[t])) for t in range(len(ids))]
        np.testing.assert_array_equal(slots, want)
        assert g.status() == 0
    finally:
        g.close()


def test_async_step_gathers_the_previous_steps_ids(weights):
    """eng_step_async: tokens whose ids the host does not know yet take, on the device, the ids the previous
    step sampled.  Two engines run the same steps, one with the ids read back on the host (eng_step), one
    with placeholders and a row map (eng_step_async): ids and logits agree bit for bit, in a replayed decode
    step, in a mixed step (a new prompt chunk plus gathered decode rows), and in a device-resident step
    after an async one.  The oracle's gather rule ("33. Removing overhead", §Async scheduling) gives the
    ids each async step reads, and its forward on those ids matches the async engine's logits and ids."""
    import torch
    from graph_replayed_decode_gb300 import eng
    from graph_replayed_decode_gb300.eng import StepArrays
    a, b = _engine(weights), _engine(weights)
    try:
        for g in (a, b):
            g.capture([1, 2, 4, 8])
        lens = [16, 9, 20]
        blocks = [list(a.alloc(3)) for _ in lens] + [list(a.alloc(2))]
        assert [list(b.alloc(3)) for _ in lens] + [list(b.alloc(2))] == blocks
        bt = block_table(blocks, MBS)
        temps = np.array([0.0, 0.9, 0.7], dtype=np.float32)
        ids = np.concatenate([synth.prompt_ids(n, S.vocab, 60 + r) for r, n in enumerate(lens)])
        pos = np.concatenate([np.arange(n) for n in lens])
        cu = np.concatenate([[0], np.cumsum(lens)])
        model = oracle.OracleModel(S, weights)
        cache = oracle.PagedCache(S, NB)
        for r, blk in enumerate(blocks):
            cache.set_block_table(r, blk)
        st1 = StepArrays(ids, pos, cu, bt[:3], np.array(lens), temps, seed=4, offset=0)
        ia, _ = a.step(st1)
        ib, lb = b.step(st1)
        np.testing.assert_array_equal(ia, ib)
        check_logits_and_ids(lb, ib, oracle.forward_step(model, cache, ids, pos, cu), temps, 4, 0)
        # decode step: explicit ids on engine a, placeholders (invalid ids, ignored) gathered on engine b
        p2 = np.array(lens)
        ia2, la2 = a.step(StepArrays(ia, p2, np.arange(4), bt[:3], p2 + 1, temps, seed=4, offset=1))
        ib2, lb2 = b.step_async(StepArrays(np.full(3, -5), p2, np.arange(4), bt[:3], p2 + 1, temps, seed=4, offset=1),
                                [0, 1, 2])
        assert b.info().replayed == 1
        np.testing.assert_array_equal(ia2, ib2)
        np.testing.assert_array_equal(la2.view(np.uint32), lb2.view(np.uint32))
        g2 = oracle.gather_input_ids(np.full(3, -5), [0, 1, 2], ib)
        np.testing.assert_array_equal(g2, ia)
        check_logits_and_ids(lb2, ib2, oracle.forward_step(model, cache, g2, p2, np.arange(4)), temps, 4, 1)
        # mixed step: a new 5-token prompt chunk (explicit ids) first, then the three decode rows; row 1's id
        # given explicitly, rows 0 and 2 gathered from the previous step's rows 0 and 2
        newp = synth.prompt_ids(5, S.vocab, 70)
        p3 = p2 + 1
        ids_a = np.concatenate([newp, ia2])
        ids_b = np.concatenate([newp, [-1, ia2[1], -1]])
        prev = np.concatenate([np.full(5, -1), [0, -1, 2]])
        pos3 = np.concatenate([np.arange(5), p3])
        cu3 = np.array([0, 5, 6, 7, 8])
        bt3 = np.concatenate([bt[3:4], bt[:3]])
        seq3 = np.concatenate([[5], p3 + 1])
        t3 = np.concatenate([[0.0], temps]).astype(np.float32)
        ia3, la3 = a.step(StepArrays(ids_a, pos3, cu3, bt3, seq3, t3, seed=4, offset=2))
        ib3, lb3 = b.step_async(StepArrays(ids_b, pos3, cu3, bt3, seq3, t3, seed=4, offset=2), prev)
        np.testing.assert_array_equal(ia3, ib3)
        np.testing.assert_array_equal(la3.view(np.uint32), lb3.view(np.uint32))
        g3 = oracle.gather_input_ids(ids_b, prev, ib2)
        np.testing.assert_array_equal(g3, ids_a)
        check_logits_and_ids(lb3, ib3, oracle.forward_step(model, cache, g3, pos3, cu3, request_keys=[3, 0, 1, 2]),
                             t3, 4, 2)
        # an async decode step, then the device-resident loop continues the batch on both engines
        p4 = p3 + 1
        a.step(StepArrays(ia3[1:], p4, np.arange(4), bt[:3], p4 + 1, temps, seed=4, offset=3))
        b.step_async(StepArrays(np.zeros(3), p4, np.arange(4), bt[:3], p4 + 1, temps, seed=4, offset=3), [1, 2, 3])
        ring_a = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
        ring_b = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
        eng.eng_decode(a.h, 2, ring_a.data_ptr())
        eng.eng_decode(b.h, 2, ring_b.data_ptr())
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ring_a.cpu().numpy(), ring_b.cpu().numpy())
        assert a.status() == 0 and b.status() == 0
        # a row outside the previous step's requests, and any gather right after a capture, are refused
        p6 = p4 + 3
        bad = StepArrays(np.zeros(3), p6, np.arange(4), bt[:3], p6 + 1, temps, seed=4, offset=6)
        with pytest.raises(eng.EngError) as ei:
            b.step_async(bad, [0, 1, 3])
        assert ei.value.code == eng.ENG_EINVAL
        b.capture([1, 2, 4, 8])
        with pytest.raises(eng.EngError) as ei:
            b.step_async(bad, [0, 1, 2])
        assert ei.value.code == eng.ENG_EINVAL
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("ks,ps", [([20, 0, 5, 1, 0], [1.0, 0.6, 0.5, 0.9, 1.0]),    # a top-p-only row: keys stored
                                   ([20, 3, 5, 1, 0], [1.0, 0.6, 0.5, 0.9, 1.0])])   # none: keys drawn in the filter
def test_top_k_top_p_inside_eager_replayed_and_device_loop_steps(weights, ks, ps):
    """Per-request filters in the step ("19. Fast decode", §Sampling without the CPU): eager prefill,
    graph-replayed decode and the device-resident loop; every id equals the oracle's filtered draw from the
    step's own logits, bit for bit, rows without a filter keep the fused draw, greedy rows the argmax.  A
    step with a top-p row that has no top-k makes the LM head store every sampling key for the filter."""
    import torch
    from graph_replayed_decode_gb300 import eng
    from graph_replayed_decode_gb300.eng import StepArrays
    g = GpuEngine(S, weights, num_blocks=NB, max_reqs=8, max_tokens=128, max_blocks_per_seq=MBS,
                  sampling_filters=True)
    try:
        g.capture([1, 2, 4, 8])
        R, P, steps = 5, 12, 5
        blocks = [list(g.alloc(oracle.blocks_needed(P + steps + 2))) for _ in range(R)]
        bt = block_table(blocks, MBS)
        temps = np.array([1.0, 1.5, 0.0, 1.2, 0.9], np.float32)
        ks = np.array(ks, np.int32)
        ps = np.array(ps, np.float32)                               # row 4: no filter
        ids = np.concatenate([synth.prompt_ids(P, S.vocab, 40 + r) for r in range(R)])
        pos = np.concatenate([np.arange(P)] * R)
        cu = np.arange(R + 1) * P
        host, changed = [], 0
        for k in range(steps):
            seq = np.array([pos[cu[r + 1] - 1] + 1 for r in range(R)])
            gid, glog = g.step(StepArrays(ids, pos, cu, bt, seq, temps, seed=9, offset=k, top_k=ks, top_p=ps))
            assert g.info().replayed == int(k > 0)
            np.testing.assert_array_equal(gid, oracle.sample_filtered(glog, temps, ks, ps, 9, k))
            changed += int(np.any(gid != oracle.sample(glog, temps, 9, k)))
            host.append(gid.copy())
            ids, pos, cu = gid.copy(), seq.copy(), np.arange(R + 1)
        assert changed > 0                                          # the filters did act on some draw
        # redo step steps-2 without asking for logits (the filters still need them), then the device loop
        k = steps - 2
        again, _ = g.step(StepArrays(host[k - 1], np.full(R, P + k - 1), np.arange(R + 1), bt, np.full(R, P + k),
                                     temps, seed=9, offset=k, top_k=ks, top_p=ps), want_logits=False)
        np.testing.assert_array_equal(again, host[k])
        ring = torch.zeros((1, R), dtype=torch.int32, device="cuda")
        eng.eng_decode(g.h, 1, ring.data_ptr())
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ring[0].cpu().numpy(), host[k + 1])
        assert g.status() == 0
    finally:
        g.close()


def test_filters_need_an_engine_created_for_them(weights):
    from graph_replayed_decode_gb300 import eng
    from graph_replayed_decode_gb300.eng import StepArrays
    g = _engine(weights)
    try:
        blocks = [list(g.alloc(1))]
        bt = block_table(blocks, MBS)
        t = np.array([1.0], np.float32)
        base = dict(token_ids=[3], positions=[0], cu_seqlens=[0, 1], block_tables=bt, seq_lens=[1], temperature=t)
        g.step(StepArrays(**base, top_k=[0], top_p=[1.0]))           # inactive filters are fine
        with pytest.raises(eng.EngError, match="sampling_filters"):
            g.step(StepArrays(**base, top_k=[5]))
        with pytest.raises(eng.EngError, match="sampling_filters"):
            g.step(StepArrays(**base, top_p=[0.5]))
        with pytest.raises(eng.EngError, match="finite"):
            g.step(StepArrays(**base, top_p=[float("nan")]))
    finally:
        g.close()


def test_generate_checks_stop_ids_once_per_group(weights):
    """eng_generate ("19. Fast decode", §Host synchronizations: stop tokens checked every check_every steps,
    one sync per check, tokens after a stop trimmed) against the oracle's stop rule applied to the tokens
    eng_decode samples on an identical engine: the same tokens, each length at the request's first stop id,
    and the steps run end at the first group boundary where all have stopped."""
    import torch
    from graph_replayed_decode_gb300 import eng
    from graph_replayed_decode_gb300.eng import StepArrays
    steps, group, R, P = 24, 4, 3, 10
    engines = []
    try:
        for _ in range(2):
            g = _engine(weights)
            engines.append(g)
            g.capture([1, 2, 4, 8])
            blocks = [list(g.alloc(oracle.blocks_needed(P + steps + 4))) for _ in range(R)]
            bt = block_table(blocks, MBS)
            temps = np.array([0.9, 1.1, 0.0], np.float32)
            ids = np.concatenate([synth.prompt_ids(P, S.vocab, 60 + r) for r in range(R)])
            pos = np.concatenate([np.arange(P)] * R)
            gid, _ = g.step(StepArrays(ids, pos, np.arange(R + 1) * P, bt, np.full(R, P), temps, seed=4, offset=0))
            g.step(StepArrays(gid, np.full(R, P), np.arange(R + 1), bt, np.full(R, P + 1), temps, seed=4, offset=1))
        a, b = engines
        ring = torch.zeros((steps, R), dtype=torch.int32, device="cuda")
        eng.eng_decode(b.h, steps, ring.data_ptr())
        torch.cuda.synchronize()
        full = ring.cpu().numpy().T                                   # [R, steps]
        stops = sorted({int(full[0, 5]), int(full[1, 13])})
        first = [next((k + 1 for k in range(steps) if full[r, k] in stops), None) for r in range(R)]
        toks, lens, n = eng.eng_generate(a.h, R, steps, group, stops)
        want_toks, want_lens, want_n = oracle.stop_trim(full, stops, group, steps)
        assert n == want_n
        np.testing.assert_array_equal(lens, want_lens)
        np.testing.assert_array_equal(toks, want_toks)
        assert n == (steps if None in first else min(steps, -(-max(first) // group) * group))
        for r in range(R):
            L = first[r] if first[r] is not None else n
            assert lens[r] == L
            np.testing.assert_array_equal(toks[r, :L], full[r, :L])
            assert (toks[r, L:] == -1).all()
        if n < steps:                                                  # the batch continues where it stopped
            nxt = torch.zeros((1, R), dtype=torch.int32, device="cuda")
            eng.eng_decode(a.h, 1, nxt.data_ptr())
            torch.cuda.synchronize()
            np.testing.assert_array_equal(nxt[0].cpu().numpy(), full[:, n])
        toks, lens, n2 = eng.eng_generate(a.h, R, 3, 8, [])           # no stop ids: every step runs
        assert n2 == 3 and (lens == 3).all()
        with pytest.raises(eng.EngError):
            eng.eng_generate(a.h, R, 4, 0, [1])                         # check_every must be >= 1
        assert a.status() == 0
    finally:
        for g in engines:
            g.close()
