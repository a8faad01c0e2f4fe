#!/usr/bin/env python
"""Decode throughput of the graph-replayed fused serving step on GB300.

Default workload (one GPU): a Qwen3-0.6B-shaped decoder (28 layers, hidden 1024, 16 Q / 8 KV heads,
head_dim 128, QK-norm, intermediate 3072, vocab 151936, tied embeddings, random bf16 weights ~N(0, 0.02)),
batch 1, a 512-token prompt prefilled eagerly into a paged cache (block 16), then pure-decode steps replayed
from the captured bucket-1 CUDA graph with Gumbel-max sampling at temperature 0.8 (capture sizes
1, 2, 4, 8, 16, 32, 64).  One step = one whole forward of the decode batch (embedding, 28 layers, final
norm, LM head, sampling, in-place advance of the next step's inputs).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0).  `value` is decode tokens/s with inputs resident on the device (eng_decode:
back-to-back graph replays); `e2e` is the same metric through eng_step with host inputs copied in and the
sampled ids read back every step.  With --gpus N > 1 (torchrun) every rank runs an independent replica.
`--impl reference` times the CPU oracle on the same workload (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from graph_replayed_decode_gb300 import roofline  # noqa: E402

METRIC = "decode tokens/s and step ms at 1 GB300; achieved fraction of HBM step roofline"
CAPTURE_SIZES = [1, 2, 4, 8, 16, 32, 64]

WORKLOADS = {
    # the metric's headline configuration
    "qwen3_0p6b_b1": dict(shape="qwen3_0p6b", batch=1, contexts=[512], temperature=0.8, prefill=True,
                          text="Qwen3-0.6B-shaped decoder, batch 1 pure decode after a 512-token prefill, "
                               "paged cache (block 16), Gumbel-max T=0.8, graph-replayed (bucket 1)"),
    "qwen3_0p6b_b32": dict(shape="qwen3_0p6b", batch=32, contexts=None, temperature=1.0, prefill=False,
                           text="Qwen3-0.6B-shaped decoder, batch 32 pure decode, contexts drawn from "
                                "{16,64,256,1024,4096} (seed 0, synthetic KV), Gumbel-max T=1.0, bucket 32"),
    "dense_8b_b64": dict(shape="dense_8b", batch=64, contexts=[2048] * 64, temperature=0.7, prefill=False,
                         text="8B-shaped dense decoder, batch 64 pure decode at context 2048 (synthetic KV), "
                              "Gumbel-max T=0.7, bucket 64"),
    # profiling case: the batch-32 kernels on a 2.5 GB device footprint (small enough for ncu captures)
    "qwen3_0p6b_b32_ctx256": dict(shape="qwen3_0p6b", batch=32, contexts=[256] * 32, temperature=1.0, prefill=False,
                                  text="Qwen3-0.6B-shaped decoder, batch 32 pure decode at context 256 "
                                       "(synthetic KV), Gumbel-max T=1.0, bucket 32"),
}

# the mixed packed step (reported under "extra" by the default run; not graph-replayed): a 512-position chunk
# of fresh prompts, then 32 decode rows
MIXED = dict(shape="qwen2p5_1p5b",
             text="Qwen2.5-1.5B-shaped decoder, one packed step: a 512-position chunk of fresh prompts "
                  "({16,64,256,1024,4096}, FCFS, the last one cut) followed by 32 decode rows at contexts from "
                  "{64,256,1024,4096} (synthetic KV), greedy, eager")


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def workload_contexts(wl: dict) -> list[int]:
    if wl["contexts"] is not None:
        return list(wl["contexts"])
    return [int(x) for x in synth.context_lengths(wl["batch"], (16, 64, 256, 1024, 4096), key=0, seed=0)]


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        # the raw samples (the JSON line carries their summary); BENCH_CLOCKS_DIR picks where they go
        out_dir = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{device_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ the CPU oracle (baseline / reference arm)


def oracle_decode_rate(wl: dict, budget_s: float, max_steps: int | None = None, warmup: int = 0) -> dict:
    """Time the CPU oracle (float64 numpy, as it stands) on decode steps of the workload.

    Setup (untimed): widened weights and each request's context filled with the same synthetic K/V
    recipe as the GPU's synthetic contexts (the 512-token prompt's cache for the batch-1 workload).
    Steps run until `budget_s` of measured time or `max_steps` steps.
    """
    import oracle
    s = synth.shape(wl["shape"])
    w = synth.make_weights(s, seed=0)
    model = oracle.OracleModel(s, w)
    B = wl["batch"]
    ctxs = workload_contexts(wl)
    rows = list(range(min(B, 4)))                  # a bounded sample of the batch: rows are independent
    room = (max_steps or 512) + warmup + 2
    cap = {r: ctxs[r] + room for r in rows}
    cache = oracle.ContiguousCache(s, cap)
    for r in rows:
        for l in range(s.layers):
            kv = synth.kv_context(s, l, r, ctxs[r])
            cache.keys[(l, r)][:, :ctxs[r], :] = oracle.widen_bf16(kv[0])
            cache.values[(l, r)][:, :ctxs[r], :] = oracle.widen_bf16(kv[1])
    ids = synth.decode_ids(len(rows), s.vocab, 0)
    pos = np.array([ctxs[r] for r in rows])
    temps = np.full(len(rows), wl["temperature"], dtype=np.float32)
    model.get("model.embed_tokens.weight")
    done, t_meas, k = 0, 0.0, 0
    while True:
        t0 = time.perf_counter()
        z = oracle.forward_step(model, cache, ids, pos, np.arange(len(rows) + 1), request_keys=rows)
        ids = oracle.sample(z.astype(np.float32), temps, 0, k)
        dt = time.perf_counter() - t0
        pos = pos + 1
        k += 1
        if k > warmup:
            done += 1
            t_meas += dt
        if max_steps is not None and done >= max_steps:
            break
        if max_steps is None and ((t_meas >= budget_s and done >= 2) or k + 1 >= room):
            break
    tokens = done * len(rows)
    return {"value": tokens / t_meas, "steps": done, "rows": len(rows), "seconds": t_meas,
            "cores": blas_threads()}


def blas_threads() -> int:
    """Threads the oracle's numpy linear algebra runs on (its matrix products are where it spends its time)."""
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 0) for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


# ------------------------------------------------------------------ our arm


class _CudaArray:
    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i2", "data": (ptr, False), "version": 3,
                                         "strides": None}


def fill_synthetic_kv(h, s, nb: int, blocks, ctxs, dtype: str = "bf16") -> None:
    """Write each request's synthetic context K/V (synth.kv_context, 16-bit values of the engine's format)
    into the engine's paged pool."""
    import torch
    from graph_replayed_decode_gb300 import eng
    ptr, nbytes = eng.eng_kv_pool(h)
    pool = torch.as_tensor(_CudaArray(ptr, nbytes // 2), device="cuda").view(s.layers, 2, nb + 1, s.kv_heads, 16,
                                                                             s.head_dim)
    for r, (b, ctx) in enumerate(zip(blocks, ctxs)):
        pos = torch.arange(ctx, device="cuda")
        bt = torch.as_tensor(np.asarray(b, dtype=np.int64), device="cuda")
        for l in range(s.layers):
            x = torch.from_numpy(synth.kv_context(s, l, r, ctx, dtype=dtype).view(np.int16)).to("cuda")
            pool[l, :, bt[pos // 16], :, pos % 16, :] = x.permute(2, 0, 1, 3)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ ranks (one replica per GPU)
#
# N GPUs run N independent replicas of the workload: no data moves between ranks. The only collective
# work is a barrier on both sides of the timed region and the maximum of the timings over the ranks.

def rank_barrier(world: int) -> None:
    if world > 1:
        import torch
        torch.distributed.barrier()


def max_over_ranks(values, world: int, device: str = "cuda") -> list[float]:
    """Each entry's largest value over all ranks (an all-reduce with MAX); unchanged for one rank."""
    values = [float(v) for v in values]
    if world <= 1:
        return values
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu().tolist()]


def whole_job_rate(world: int, rows_per_rank: int, steps: int, seconds: float) -> float:
    """Tokens per second of the whole job: every rank samples rows_per_rank tokens per step."""
    return world * rows_per_rank * steps / seconds


def run_ours(args, wl: dict, rank: int, world: int, local_rank: int) -> dict | None:
    import torch
    torch.cuda.set_device(local_rank)
    from graph_replayed_decode_gb300 import build, eng
    if not os.path.exists(eng.LIB_PATH):
        if rank == 0:
            build.build()
        rank_barrier(world)
    s = synth.shape(wl["shape"])
    B = wl["batch"]
    ctxs = workload_contexts(wl)
    K, W = args.steps, args.warmup
    extra = 1 + W + K + 1 + args.steps + 8          # first step, warmup, timed, profile, e2e
    mbs = -(-(max(ctxs) + extra) // 16)
    need = [-(-(c + extra) // 16) for c in ctxs]
    nb = sum(need) + 8
    max_tokens = max(512 if wl["prefill"] else 64, 64)

    weights = synth.make_weights(s, seed=0, cache=False)
    stream = torch.cuda.Stream()
    filters = args.top_k > 0 or 0.0 < args.top_p < 1.0
    h = eng.eng_create(eng.make_config(s, nb, 64, max_tokens, mbs, sampling_filters=filters),
                       eng.TensorList(weights.items()), stream.cuda_stream)
    fk = dict(top_k=np.full(B, args.top_k, np.int32), top_p=np.full(B, args.top_p, np.float32)) if filters else {}
    del weights
    ids_dev = torch.zeros(64, dtype=torch.int32, device="cuda")
    temps = np.full(B, wl["temperature"], dtype=np.float32)
    blocks = [eng.eng_pool_alloc(h, n) for n in need]
    bt = np.zeros((B, mbs), dtype=np.int32)
    for r, b in enumerate(blocks):
        bt[r, :len(b)] = b
    out = {}
    # ---- context: a real eager prefill (batch 1) or synthetic K/V written into the pool
    if wl["prefill"]:
        assert B == 1
        prompt = synth.prompt_ids(ctxs[0], s.vocab, 0)
        st = eng.StepArrays(prompt, np.arange(ctxs[0]), [0, ctxs[0]], bt, [ctxs[0]], temps, seed=0, offset=0, **fk)
        eng.eng_step(h, st, ids_dev.data_ptr(), None)   # warm-up: same prompt, same blocks, same K/V written
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record()
            eng.eng_step(h, st, ids_dev.data_ptr(), None)
            e1.record()
        torch.cuda.synchronize()
        out["prefill_ms"] = e0.elapsed_time(e1)
        first = ids_dev[:1].cpu().numpy()
    else:
        fill_synthetic_kv(h, s, nb, blocks, ctxs)
        first = synth.decode_ids(B, s.vocab, 0)
    eng.eng_capture(h, CAPTURE_SIZES)

    pos = np.array(ctxs, dtype=np.int32)
    st = eng.StepArrays(first, pos, np.arange(B + 1), bt, pos + 1, temps, seed=0, offset=1, **fk)
    eng.eng_step(h, st, ids_dev.data_ptr(), None)           # first decode step (host inputs)
    launches_per_step = eng.eng_last_step_info(h).launches
    ring = torch.zeros((max(K, W, 1), B), dtype=torch.int32, device="cuda")

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    eng.eng_decode(h, W, ring.data_ptr())                     # warm-up replays
    torch.cuda.synchronize()
    rank_barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    with torch.cuda.stream(stream):
        e0.record()
        eng.eng_decode(h, K, ring.data_ptr())
        e1.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    t_dev = e0.elapsed_time(e1) / 1e3
    rank_barrier(world)
    seq_timed = [c + 1 + W + k + 1 for c in ctxs for k in range(K)]    # keys seen by each timed step's rows

    # ---- per-kernel timing of one more step (CUDA events around every launch on the engine stream)
    prof = eng.eng_profile(h)

    # ---- end to end: eng_step with host inputs and a device->host read of the sampled ids every step
    pinned = torch.zeros(B, dtype=torch.int32).pin_memory()
    ids_h = ring[K - 1].cpu().numpy() if K > 0 else first
    pos = pos + 1 + W + K + 1
    torch.cuda.synchronize()
    h2d = 0
    t0 = time.perf_counter()
    for k in range(K):
        st = eng.StepArrays(ids_h, pos, np.arange(B + 1), bt, pos + 1, temps, seed=0, offset=10_000 + k, **fk)
        eng.eng_step(h, st, ids_dev.data_ptr(), None)
        with torch.cuda.stream(stream):
            pinned.copy_(ids_dev[:B], non_blocking=True)
        stream.synchronize()
        ids_h = pinned.numpy().copy()
        pos = pos + 1
        h2d = eng.eng_last_step_info(h).h2d_bytes
    t_e2e = time.perf_counter() - t0
    clk = clocks.stop()
    status = eng.eng_status(h, True)
    eng.eng_destroy(h)

    # ---- max over ranks
    t_dev, t_e2e = max_over_ranks([t_dev, t_e2e], world)
    if rank != 0:
        return None

    peaks = load_peaks()
    bw = peaks["hbm_gbs"] * 1e9
    mean_seq = float(np.mean(seq_timed))
    step_b = roofline.step_bytes(s, B, [mean_seq] * B)
    t_roof = step_b / bw
    step_s = t_dev / K
    # dominant kernel kind by total time of the profiled step
    agg: dict[str, list] = {}
    for kind, ms, nbytes in prof:
        a = agg.setdefault(kind, [0, 0.0, 0])
        a[0] += 1
        a[1] += ms
        a[2] += nbytes
    dom = max(agg.items(), key=lambda kv: kv[1][1])
    dk, (dn, dms, dbytes) = dom
    achieved = (dbytes / dn) / (dms / dn / 1e3) / 1e9
    traffic = load_traffic(wl_name=args.workload, kind=dk)
    result = {
        "metric": METRIC,
        "value": whole_job_rate(world, B, K, t_dev),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": step_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl["text"], "batch": B, "context_start": ctxs if B <= 4 else "seeded draw",
                   "temperature": wl["temperature"], "capture_sizes": CAPTURE_SIZES,
                   **({"top_k": args.top_k, "top_p": args.top_p} if filters else {}),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {roofline.weight_bytes(s) / 1e9:.3f} GB of weights read per step"},
        "step_roofline": {"bytes_per_step": int(step_b), "t_roof_ms": t_roof * 1e3, "frac": t_roof / step_s,
                          "peak_gbs": peaks["hbm_gbs"], "of": peaks["source"]},
        "roofline": {"kernel": dk, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "launches_per_step": dn,
                     "share_of_step": dms / sum(a[1] for a in agg.values()), "of": peaks["source"]},
        "kernels": {k: {"launches": v[0], "ms": round(v[1], 4), "gbs": round(v[2] / (v[1] / 1e3) / 1e9, 1)}
                    for k, v in sorted(agg.items(), key=lambda kv: -kv[1][1])},
        "e2e": {"value": whole_job_rate(world, B, K, t_e2e), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": 4 * B},
        "gpu_launches": K * launches_per_step,
        "clocks": clk,
        "device_status": status,
    }
    if "prefill_ms" in out:
        result["prefill_ms"] = out["prefill_ms"]
    if world == 1 and not args.no_cpu_baseline:
        cb = oracle_decode_rate(wl, budget_s=args.cpu_seconds, warmup=1)
        result["cpu_baseline"] = {"value": cb["value"], "unit": "tokens/s", "cores": cb["cores"], "kind": "oracle",
                                  "sample": f"{cb['steps']} decode steps x {cb['rows']} row(s) of this workload "
                                            f"(float64 numpy oracle, synthetic context), {cb['seconds']:.1f} s"}
    return result


def run_mixed(steps: int, warmup: int, local_rank: int, dtype: str = "bf16") -> dict:
    """The mixed packed step of the Qwen2.5-1.5B workload, eager (mixed steps are not replayed): the same step
    `steps` times with host inputs (device time with CUDA events, and end to end with the sampled ids read
    back), against the step roofline max(bytes / HBM, flops / sustained bf16 tensor peak; dense fp16 has the
    same nominal rate).  dtype "f16" runs the fp16 variant of the model (fp16 weights, K/V and operands)."""
    import torch
    from graph_replayed_decode_gb300 import eng
    wl = MIXED
    s = synth.shape(wl["shape"])
    chunk = synth.mixed_chunk_prompts(512, key=0, seed=0)
    P = len(chunk)
    dctx = [int(c) for c in synth.context_lengths(32, (64, 256, 1024, 4096), key=1, seed=0)]
    need = [-(-(plen + 1) // 16) for plen, _ in chunk] + [-(-(c + 1) // 16) for c in dctx]
    mbs = max(need)
    nb = sum(need) + 4
    weights = synth.make_weights(s, seed=0, cache=False, dtype=dtype)
    stream = torch.cuda.Stream()
    h = eng.eng_create(eng.make_config(s, nb, 64, 600, mbs, dtype=dtype), eng.TensorList(weights.items(), dtype),
                       stream.cuda_stream)
    del weights
    blocks = [eng.eng_pool_alloc(h, n) for n in need]
    bt = np.zeros((P + 32, mbs), dtype=np.int32)
    for r, b in enumerate(blocks):
        bt[r, :len(b)] = b
    fill_synthetic_kv(h, s, nb, blocks[P:], dctx, dtype)
    prompts = [synth.prompt_ids(take, s.vocab, 50 + i) for i, (plen, take) in enumerate(chunk)]
    ids = np.concatenate(prompts + [synth.decode_ids(32, s.vocab, 2)]).astype(np.int32)
    pos = np.concatenate([np.arange(take) for _, take in chunk] + [np.array(dctx)]).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum([take for _, take in chunk] + [1] * 32)]).astype(np.int32)
    seq = np.array([take for _, take in chunk] + [c + 1 for c in dctx], dtype=np.int32)
    temps = np.zeros(P + 32, dtype=np.float32)
    st = eng.StepArrays(ids, pos, cu, bt, seq, temps, seed=0, offset=0)
    ids_dev = torch.zeros(64, dtype=torch.int32, device="cuda")
    T = int(cu[-1])
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    for _ in range(warmup):
        eng.eng_step(h, st, ids_dev.data_ptr(), None)
    torch.cuda.synchronize()
    launches = eng.eng_last_step_info(h).launches
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(steps):
            eng.eng_step(h, st, ids_dev.data_ptr(), None)
        e1.record()
    torch.cuda.synchronize()
    t_dev = e0.elapsed_time(e1) / 1e3 / steps
    pinned = torch.zeros(P + 32, dtype=torch.int32).pin_memory()
    t0 = time.perf_counter()
    for _ in range(steps):
        eng.eng_step(h, st, ids_dev.data_ptr(), None)
        with torch.cuda.stream(stream):
            pinned.copy_(ids_dev[:P + 32], non_blocking=True)
        stream.synchronize()
    t_e2e = (time.perf_counter() - t0) / steps
    h2d = eng.eng_last_step_info(h).h2d_bytes
    # the same step on piecewise graphs: the projections of a bucket of the step's token count replayed,
    # attention between
    eng.eng_capture_mixed(h, [T])
    for _ in range(warmup):
        eng.eng_step(h, st, ids_dev.data_ptr(), None)
    torch.cuda.synchronize()
    assert eng.eng_last_step_info(h).replayed == 2
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(steps):
            eng.eng_step(h, st, ids_dev.data_ptr(), None)
        e1.record()
    torch.cuda.synchronize()
    t_pw = e0.elapsed_time(e1) / 1e3 / steps
    clk = clocks.stop()
    status = eng.eng_status(h, True)
    eng.eng_destroy(h)
    peaks = load_peaks()
    keys_seen = sum(take * (take + 1) // 2 for _, take in chunk) + sum(c + 1 for c in dctx)
    flops = roofline.step_flops(s, T, P + 32, keys_seen)
    nbytes = roofline.step_bytes(s, T, [int(x) for x in seq])
    t_b = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_f = flops / (peaks["bf16_tflops_sustained"] * 1e12)
    text = wl["text"] if dtype == "bf16" else wl["text"].replace("Qwen2.5-1.5B-shaped decoder", "Qwen2.5-1.5B-shaped decoder in fp16")
    return {"workload": text, "dtype": dtype, "tokens_per_step": T, "requests": P + 32, "steps": steps, "warmup": warmup,
            "ms_per_step": t_dev * 1e3, "value": T / t_dev, "unit": "tokens/s",
            "step_roofline": {"bound": "tensor" if t_f >= t_b else "hbm", "bytes_per_step": int(nbytes),
                              "flops_per_step": int(flops), "t_roof_ms": max(t_b, t_f) * 1e3,
                              "frac": max(t_b, t_f) / t_dev, "achieved_tflops": flops / t_dev / 1e12,
                              "peak_tflops": peaks["bf16_tflops_sustained"], "peak_gbs": peaks["hbm_gbs"],
                              "of": peaks["source"] + " (sustained bf16 for the tensor bound)"},
            "e2e": {"value": T / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": 4 * (P + 32)},
            "piecewise": {"ms_per_step": t_pw * 1e3, "value": T / t_pw, "unit": "tokens/s",
                          "frac": max(t_b, t_f) / t_pw, "bucket_tokens": T,
                          "note": "projection pieces replayed as graphs, attention and LM head launched between"},
            "gpu_launches": steps * launches, "clocks": clk, "device_status": status}


def run_moe(steps: int, warmup: int) -> dict:
    """The Qwen3-30B-A3B-shaped mixture-of-experts layer (eng_moe_mlp: alignment, grouped gate|up and down
    GEMMs, combine) at a decode batch (32 tokens) and a prefill chunk (512 tokens), routed by the oracle's
    router on synthetic token rows.  Step roofline: the experts' weights that the routing touches plus the
    token rows in and the outputs, over measured HBM bandwidth (flops / sustained bf16 peak is smaller)."""
    import torch
    from graph_replayed_decode_gb300 import eng
    import oracle.moe as omoe
    from oracle.model import widen_bf16
    m = synth.moe_shape("qwen3_30b_a3b_moe")
    w = synth.moe_weights(m, seed=0)
    peaks = load_peaks()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    gu, dn = dev(w["gate_up"]), dev(w["down"])
    out = {"workload": "Qwen3-30B-A3B-shaped MoE MLP: hidden 2048, 128 experts, 8 per token, expert width 768, "
                       "bf16 weights, routed by the oracle's router on synthetic token rows"}
    for N in (32, 512):
        x = synth.moe_tokens(N, m.hidden, key=7)
        rw, ids = omoe.route(widen_bf16(x), widen_bf16(w["router"]), m.top_k)
        dx = dev(x)
        drw = torch.from_numpy(rw.astype(np.float32)).cuda()
        dids = torch.from_numpy(ids.astype(np.int32)).cuda()
        y = torch.empty((N, m.hidden), dtype=torch.float32, device="cuda")
        nbytes = eng.eng_moe_workspace_bytes(N, m.top_k, m.experts, m.hidden, m.intermediate)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")  # larger than L2, between calls
        call = lambda: eng.eng_moe_mlp(dx.data_ptr(), gu.data_ptr(), dn.data_ptr(), drw.data_ptr(), dids.data_ptr(), N,
                                       m.hidden, m.intermediate, m.experts, m.top_k, y.data_ptr(), ws.data_ptr(),
                                       nbytes, torch.cuda.current_stream().cuda_stream)
        for _ in range(warmup):
            call()
        times = []
        for _ in range(steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / 1e3)
        t = statistics.median(times)
        used = len(np.unique(ids))
        nbytes_alg = used * (2 * m.intermediate * m.hidden + m.hidden * m.intermediate) * 2 + N * m.hidden * (2 + 4)
        flops = 2 * N * m.top_k * 3 * m.intermediate * m.hidden
        t_roof = max(nbytes_alg / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops_sustained"] * 1e12))
        out[f"tokens_{N}"] = {"ms": t * 1e3, "experts_touched": used, "bytes": int(nbytes_alg), "flops": int(flops),
                              "achieved_gbs": nbytes_alg / t / 1e9, "t_roof_ms": t_roof * 1e3, "frac": t_roof / t,
                              "bound": "hbm", "peak_gbs": peaks["hbm_gbs"], "of": peaks["source"],
                              "timing": f"median of {steps} calls, L2 flushed (256 MB written) before each"}
    return out


def run_extras(args, local_rank: int) -> dict:
    """The other configurations the metric is stated on, in the same run: batch-32 decode (graph-replayed)
    and the mixed packed step (bf16, and its fp16 variant), each with its own roofline, clocks and end-to-end
    figure; and the mixture-of-experts layer of the MoE calls."""
    import copy
    out = {}
    a = copy.copy(args)
    a.steps, a.warmup, a.workload, a.no_cpu_baseline = min(args.steps, 64), min(args.warmup, 8), "qwen3_0p6b_b32", True
    r = run_ours(a, WORKLOADS["qwen3_0p6b_b32"], 0, 1, local_rank)
    out["qwen3_0p6b_b32"] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "config",
                                                "step_roofline", "roofline", "e2e", "gpu_launches", "clocks",
                                                "device_status")}
    out["qwen3_0p6b_b32"]["kernels"] = dict(list(r["kernels"].items())[:4])
    out["qwen2p5_1p5b_mixed"] = run_mixed(min(args.steps, 16), min(args.warmup, 4), local_rank)
    out["qwen2p5_1p5b_mixed_f16"] = run_mixed(min(args.steps, 16), min(args.warmup, 4), local_rank, dtype="f16")
    out["qwen3_30b_a3b_moe_layer"] = run_moe(min(args.steps, 20), 3)
    return out


def load_traffic(wl_name: str, kind: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    entry = d.get(wl_name, {}).get(kind)
    if not entry or entry.get("sources_hash") != sources_hash():
        return None
    return entry.get("bytes_per_launch")


def sources_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "graph_replayed_decode_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="qwen3_0p6b_b1")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--top-k", type=int, default=0, help="top-k filter on every row (0: off)")
    ap.add_argument("--top-p", type=float, default=1.0, help="top-p filter on every row (1: off)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the batch-32 and mixed-step figures that the default run adds under 'extra'")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    wl = WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        r = oracle_decode_rate(wl, budget_s=0.0, max_steps=args.steps, warmup=max(args.warmup, 1))
        line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["seconds"] / max(r["steps"], 1) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": wl["text"], "batch": wl["batch"],
                           "context_start": workload_contexts(wl) if wl["batch"] <= 4 else "seeded draw",
                           "temperature": wl["temperature"],
                           "sample": f"CPU oracle, {r['rows']} of the batch's rows per step"},
                "cpu_baseline": {"value": r["value"], "unit": "tokens/s", "cores": r["cores"], "kind": "oracle",
                                 "sample": f"{r['steps']} timed decode steps x {r['rows']} row(s), float64 numpy"},
                "e2e": {"value": r["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, wl, rank, world, local_rank)
    if res is not None and world == 1 and args.workload == "qwen3_0p6b_b1" and not args.no_extra:
        res["extra"] = run_extras(args, local_rank)
    if res is not None:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
