"""Test helpers: drive libeng.so (through its C-ABI binding) and the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import os

import numpy as np

import synth

TOL_LOGITS = 3e-2      # max-abs logit error, bf16 weights/activations with fp32 accumulation
GREEDY_MARGIN = 0.1    # greedy ids must agree where the oracle's top-2 margin exceeds this


def ensure_built():
    from graph_replayed_decode_gb300 import build, eng
    if not os.path.exists(eng.LIB_PATH):
        build.build()
    return eng


class _CudaArray:
    """Minimal __cuda_array_interface__ so torch can view engine-owned device memory."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def device_view(ptr: int, nbytes: int, dtype):
    import torch
    typestr = {torch.int16: "<i2", torch.int32: "<i4", torch.float32: "<f4"}[dtype]
    item = {torch.int16: 2, torch.int32: 4, torch.float32: 4}[dtype]
    return torch.as_tensor(_CudaArray(ptr, (nbytes // item,), typestr), device="cuda")


class GpuEngine:
    """One engine over synth weights; outputs come back as numpy arrays."""

    def __init__(self, s: synth.ModelShape, weights, num_blocks: int, max_reqs: int, max_tokens: int,
                 max_blocks_per_seq: int, stream=None, sampling_filters: bool = False):
        import torch
        self.eng = ensure_built()
        self.torch = torch
        self.s = s
        self.num_blocks = num_blocks
        self.max_blocks_per_seq = max_blocks_per_seq
        dtype = getattr(weights, "dtype", "bf16")  # synth weights name their 16-bit format
        cfg = self.eng.make_config(s, num_blocks, max_reqs, max_tokens, max_blocks_per_seq, sampling_filters, dtype)
        tl = self.eng.TensorList(weights.items(), dtype)
        self.stream = stream
        self.h = self.eng.eng_create(cfg, tl, None if stream is None else stream.cuda_stream)
        del tl
        self.ids_dev = torch.zeros(max_reqs, dtype=torch.int32, device="cuda")
        self.logits_dev = torch.zeros((max_reqs, s.vocab), dtype=torch.float32, device="cuda")

    def close(self):
        if self.h is not None:
            self.eng.eng_destroy(self.h)
            self.h = None

    def capture(self, sizes):
        self.eng.eng_capture(self.h, sizes)

    def capture_mixed(self, token_buckets):
        self.eng.eng_capture_mixed(self.h, token_buckets)

    def alloc(self, n):
        return self.eng.eng_pool_alloc(self.h, n)

    def kv_pool(self):
        """torch int16 view [L, 2, NB+1, Hkv, 16, d] of the engine's KV pool (16-bit bits of the model's format)."""
        ptr, nbytes = self.eng.eng_kv_pool(self.h)
        s = self.s
        return device_view(ptr, nbytes, self.torch.int16).view(s.layers, 2, self.num_blocks + 1, s.kv_heads, 16,
                                                              s.head_dim)

    def fill_context(self, layer: int, blocks, kv_bits: np.ndarray):
        """Write synthetic K/V [2, Hkv, ctx, d] (16-bit bits) of positions 0..ctx-1 through a block table."""
        torch = self.torch
        ctx = kv_bits.shape[2]
        pool = self.kv_pool()
        pos = torch.arange(ctx, device="cuda")
        bt = torch.as_tensor(np.asarray(blocks, dtype=np.int64), device="cuda")
        x = torch.from_numpy(np.ascontiguousarray(kv_bits).view(np.int16)).to("cuda")
        pool[layer, :, bt[pos // 16], :, pos % 16, :] = x.permute(2, 0, 1, 3)

    def step(self, step, want_logits: bool = True):
        torch = self.torch
        R = len(step.cu_seqlens) - 1
        self.eng.eng_step(self.h, step, self.ids_dev.data_ptr(), self.logits_dev.data_ptr() if want_logits else None)
        torch.cuda.synchronize()
        ids = self.ids_dev[:R].cpu().numpy().copy()
        logits = self.logits_dev[:R].cpu().numpy().copy() if want_logits else None
        return ids, logits

    def step_async(self, step, prev_row, want_logits: bool = True):
        torch = self.torch
        R = len(step.cu_seqlens) - 1
        self.eng.eng_step_async(self.h, step, prev_row, self.ids_dev.data_ptr(),
                                self.logits_dev.data_ptr() if want_logits else None)
        torch.cuda.synchronize()
        ids = self.ids_dev[:R].cpu().numpy().copy()
        logits = self.logits_dev[:R].cpu().numpy().copy() if want_logits else None
        return ids, logits

    def info(self):
        return self.eng.eng_last_step_info(self.h)

    def status(self, reset=True):
        return self.eng.eng_status(self.h, reset)


def block_table(blocks_per_req, width):
    bt = np.zeros((len(blocks_per_req), width), dtype=np.int32)
    for r, b in enumerate(blocks_per_req):
        bt[r, :len(b)] = b
    return bt


def check_logits_and_ids(gpu_logits, gpu_ids, oracle_logits, temps, seed, offset, rows=None, tol=TOL_LOGITS):
    """The parity bar: logits within tol, ids re-sampled from the GPU's own logits bit-exact, and
    greedy rows equal to the oracle's argmax wherever its top-2 margin exceeds GREEDY_MARGIN."""
    import oracle
    rows = list(range(gpu_logits.shape[0])) if rows is None else list(rows)
    err = np.abs(gpu_logits[rows].astype(np.float64) - oracle_logits).max()
    assert err <= tol, f"max-abs logit error {err} > {tol}"
    for i, r in enumerate(rows):
        z = gpu_logits[r].astype(np.float32)
        want = oracle.sample_row(z, float(temps[r]), seed, offset, r)
        assert gpu_ids[r] == want, (r, gpu_ids[r], want)
        if temps[r] == 0.0:
            srt = np.sort(oracle_logits[i])
            if srt[-1] - srt[-2] > GREEDY_MARGIN:
                assert gpu_ids[r] == int(np.argmax(oracle_logits[i]))
    return err
