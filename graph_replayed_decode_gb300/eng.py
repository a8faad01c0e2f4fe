"""ctypes binding of libeng.so, one Python function per C entry point of include/eng.h.

Argument marshalling only: every step of the forward runs in the library's CUDA
kernels.  Loading fails loudly if the library has not been built (there is no
CPU fallback).  Device pointers are plain integers (for example
``torch.Tensor.data_ptr()``); host arrays are numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Sequence

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libeng.so")

ENG_OK = 0
ENG_EINVAL = -1
ENG_ECAPACITY = -2
ENG_ENOMEM = -3
ENG_EPOOL = -4
ENG_ECUDA = -5
ENG_EDEVICE = -6
ENG_ESTATE = -7

ENG_STATUS_BAD_BLOCK = 1
ENG_STATUS_BAD_POSITION = 2
ENG_STATUS_NAN = 4
ENG_STATUS_TIMEOUT = 8

ENG_DTYPE_BF16 = 0
ENG_DTYPE_F16 = 1
ENG_DTYPE_F32 = 2


class eng_config_t(ctypes.Structure):
    _fields_ = [
        ("layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("q_heads", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
        ("qk_norm", ctypes.c_int32), ("qkv_bias", ctypes.c_int32), ("tie_embeddings", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("max_reqs", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
        ("sampling_filters", ctypes.c_int32),
    ]


class eng_tensor_t(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("data", ctypes.c_void_p), ("numel", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("on_device", ctypes.c_int32)]


_I32P = ctypes.POINTER(ctypes.c_int32)
_F32P = ctypes.POINTER(ctypes.c_float)


class eng_step_t(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_reqs", ctypes.c_int32), ("bt_stride", ctypes.c_int32),
                ("token_ids", _I32P), ("positions", _I32P), ("cu_seqlens", _I32P), ("block_tables", _I32P),
                ("seq_lens", _I32P), ("temperature", _F32P), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
                ("top_k", _I32P), ("top_p", _F32P)]


class eng_step_info_t(ctypes.Structure):
    _fields_ = [("replayed", ctypes.c_int32), ("bucket", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("num_prefill", ctypes.c_int32), ("h2d_bytes", ctypes.c_int64)]


class EngError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


_lib = None

# (name, restype, argtypes) of every entry point declared in include/eng.h
SIGNATURES = [
    ("eng_create", ctypes.c_int, [ctypes.POINTER(eng_config_t), ctypes.POINTER(eng_tensor_t), ctypes.c_int32,
                                  ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    ("eng_capture", ctypes.c_int, [ctypes.c_void_p, _I32P, ctypes.c_int32]),
    ("eng_capture_mixed", ctypes.c_int, [ctypes.c_void_p, _I32P, ctypes.c_int32]),
    ("eng_step", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(eng_step_t), ctypes.c_void_p, ctypes.c_void_p]),
    ("eng_step_async", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(eng_step_t), ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    ("eng_last_step_info", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(eng_step_info_t)]),
    ("eng_decode", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    ("eng_profile", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _I32P, _F32P, ctypes.POINTER(ctypes.c_int64),
                                   _I32P]),
    ("eng_pool_alloc", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, _I32P]),
    ("eng_pool_free", ctypes.c_int, [ctypes.c_void_p, _I32P, ctypes.c_int32]),
    ("eng_pool_free_count", ctypes.c_int32, [ctypes.c_void_p]),
    ("eng_status", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("eng_set_eager", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    ("eng_kv_pool", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int64)]),
    ("eng_debug_buffer", ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_void_p),
                                        ctypes.POINTER(ctypes.c_int64)]),
    ("eng_stream", ctypes.c_void_p, [ctypes.c_void_p]),
    ("eng_last_error", ctypes.c_char_p, [ctypes.c_void_p]),
    ("eng_destroy", None, [ctypes.c_void_p]),
    ("eng_philox_uniforms", ctypes.c_int, [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_void_p]),
    ("eng_gumbel", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
    ("eng_sample", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, _F32P, ctypes.c_uint64,
                                  ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]),
    ("eng_sample_noalloc", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, _F32P, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]),
    ("eng_sample_filtered", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, _F32P,
                                           _I32P, _F32P, ctypes.c_uint64, ctypes.c_uint64,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    ("eng_exp_f32", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
    ("eng_generate", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, _I32P, ctypes.c_int32, _I32P,
                                    _I32P]),
    ("eng_moe_route", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    ("eng_moe_padded_rows", ctypes.c_int64, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    ("eng_moe_align", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    ("eng_moe_workspace_bytes", ctypes.c_int64, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32]),
    ("eng_moe_mlp", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
]


def lib() -> ctypes.CDLL:
    """The loaded libeng.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built (python -m graph_replayed_decode_gb300.build); "
                               "the engine has no CPU fallback")
        l = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _check(e, rc: int) -> int:
    if rc < 0:
        msg = lib().eng_last_error(e)
        raise EngError(rc, msg.decode() if msg else "")
    return rc


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(_I32P)


# ------------------------------------------------------------------ marshalling helpers


def make_config(shape, num_blocks: int, max_reqs: int, max_tokens: int, max_blocks_per_seq: int,
                sampling_filters: bool = False, dtype: str = "bf16") -> eng_config_t:
    """eng_config_t from a model shape (any object with the synth.ModelShape fields); dtype "bf16" or "f16"
    names the 16-bit format of the weights and activations."""
    if dtype not in ("bf16", "f16"):
        raise ValueError(f"dtype must be 'bf16' or 'f16', not {dtype!r}")
    return eng_config_t(
        layers=shape.layers, hidden=shape.hidden, q_heads=shape.q_heads, kv_heads=shape.kv_heads,
        head_dim=shape.head_dim, intermediate=shape.intermediate, vocab=shape.vocab, rms_eps=shape.rms_eps,
        rope_theta=shape.rope_theta, qk_norm=int(shape.qk_norm), qkv_bias=int(shape.qkv_bias),
        tie_embeddings=int(shape.tie_embeddings), dtype=ENG_DTYPE_BF16 if dtype == "bf16" else ENG_DTYPE_F16,
        block_size=16, num_blocks=num_blocks,
        max_reqs=max_reqs, max_tokens=max_tokens, max_blocks_per_seq=max_blocks_per_seq,
        sampling_filters=int(sampling_filters))


class TensorList:
    """eng_tensor_t array over host numpy arrays (16-bit values as uint16 bits, of the format dtype names:
    "bf16" or "f16") that keeps them alive."""

    def __init__(self, items: Iterable[tuple[str, np.ndarray]], dtype: str = "bf16"):
        if dtype not in ("bf16", "f16"):
            raise ValueError(f"dtype must be 'bf16' or 'f16', not {dtype!r}")
        self._keep = []
        recs = []
        for name, arr in items:
            arr = np.ascontiguousarray(arr)
            if arr.dtype == np.uint16:
                dt = ENG_DTYPE_BF16 if dtype == "bf16" else ENG_DTYPE_F16
            elif arr.dtype == np.float32:
                dt = ENG_DTYPE_F32
            else:
                raise TypeError(f"{name}: weights are 16-bit bits (uint16) or float32")
            nm = name.encode()
            self._keep += [arr, nm]
            recs.append(eng_tensor_t(nm, arr.ctypes.data, arr.size, dt, 0))
        self.array = (eng_tensor_t * len(recs))(*recs)
        self.count = len(recs)


class StepArrays:
    """eng_step_t over host arrays (kept alive by this object)."""

    def __init__(self, token_ids, positions, cu_seqlens, block_tables, seq_lens, temperature, seed: int = 0,
                 offset: int = 0, top_k=None, top_p=None):
        self.token_ids = _i32(token_ids)
        self.positions = _i32(positions)
        self.cu_seqlens = _i32(cu_seqlens)
        bt = np.atleast_2d(_i32(block_tables))
        self.block_tables = np.ascontiguousarray(bt)
        self.seq_lens = _i32(seq_lens)
        self.temperature = np.ascontiguousarray(temperature, dtype=np.float32)
        self.top_k = None if top_k is None else _i32(top_k)
        self.top_p = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32)
        R = len(self.cu_seqlens) - 1
        self.step = eng_step_t(
            num_tokens=len(self.token_ids), num_reqs=R, bt_stride=self.block_tables.shape[1],
            token_ids=_ptr_i32(self.token_ids), positions=_ptr_i32(self.positions),
            cu_seqlens=_ptr_i32(self.cu_seqlens), block_tables=_ptr_i32(self.block_tables),
            seq_lens=_ptr_i32(self.seq_lens), temperature=self.temperature.ctypes.data_as(_F32P),
            seed=int(seed), offset=int(offset),
            top_k=None if self.top_k is None else _ptr_i32(self.top_k),
            top_p=None if self.top_p is None else self.top_p.ctypes.data_as(_F32P))


# ------------------------------------------------------------------ entry points


def eng_create(cfg: eng_config_t, weights: TensorList, cuda_stream: int | None = None) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    rc = lib().eng_create(ctypes.byref(cfg), weights.array, weights.count, cuda_stream, ctypes.byref(h))
    _check(None, rc)
    return h


def eng_capture(e, sizes: Sequence[int]) -> None:
    s = _i32(sizes)
    _check(e, lib().eng_capture(e, _ptr_i32(s), len(s)))


def eng_capture_mixed(e, token_buckets: Sequence[int]) -> None:
    """Piecewise graphs of the projections of mixed steps, one set per token bucket."""
    s = _i32(token_buckets)
    _check(e, lib().eng_capture_mixed(e, _ptr_i32(s), len(s)))


def eng_step(e, step: StepArrays, out_ids_dev: int, out_logits_dev: int | None = None) -> None:
    _check(e, lib().eng_step(e, ctypes.byref(step.step), out_ids_dev, out_logits_dev))


def eng_step_async(e, step: StepArrays, prev_row, out_ids_dev: int, out_logits_dev: int | None = None) -> None:
    """eng_step where token t with prev_row[t] = r >= 0 takes the id the previous step sampled for row r."""
    pr = np.ascontiguousarray(prev_row, dtype=np.int32)
    if pr.shape != (step.step.num_tokens,):
        raise ValueError("prev_row needs one entry per token")
    _check(e, lib().eng_step_async(e, ctypes.byref(step.step), pr.ctypes.data, out_ids_dev, out_logits_dev))


def eng_last_step_info(e) -> eng_step_info_t:
    info = eng_step_info_t()
    _check(e, lib().eng_last_step_info(e, ctypes.byref(info)))
    return info


def eng_decode(e, n_steps: int, out_ids_dev: int) -> None:
    _check(e, lib().eng_decode(e, n_steps, out_ids_dev))


KERNEL_KINDS = ["embed_norm", "norm", "gemm_qkv", "rope_kv", "attn_decode", "attn_prefill", "gemm_o",
                "gemm_gate_up", "gemm_down", "lm_head", "advance", "sample_filter", "decode_layers"]


def eng_profile(e, capacity: int = 4096):
    """Per-launch (kind name, ms, algorithmic bytes) of one further decode step."""
    kinds = np.zeros(capacity, dtype=np.int32)
    ms = np.zeros(capacity, dtype=np.float32)
    nbytes = np.zeros(capacity, dtype=np.int64)
    n = ctypes.c_int32()
    _check(e, lib().eng_profile(e, capacity, _ptr_i32(kinds), ms.ctypes.data_as(_F32P),
                                nbytes.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ctypes.byref(n)))
    k = n.value
    return [(KERNEL_KINDS[kinds[i]], float(ms[i]), int(nbytes[i])) for i in range(k)]


def eng_pool_alloc(e, n: int) -> np.ndarray:
    out = np.zeros(max(n, 1), dtype=np.int32)
    _check(e, lib().eng_pool_alloc(e, n, _ptr_i32(out)))
    return out[:n]


def eng_pool_free(e, ids) -> None:
    a = _i32(ids)
    _check(e, lib().eng_pool_free(e, _ptr_i32(a), len(a)))


def eng_pool_free_count(e) -> int:
    return int(lib().eng_pool_free_count(e))


def eng_status(e, reset: bool = False) -> int:
    return _check(e, lib().eng_status(e, int(reset)))


def eng_set_eager(e, eager: bool) -> None:
    _check(e, lib().eng_set_eager(e, int(eager)))


def eng_kv_pool(e) -> tuple[int, int]:
    p = ctypes.c_void_p()
    n = ctypes.c_int64()
    _check(e, lib().eng_kv_pool(e, ctypes.byref(p), ctypes.byref(n)))
    return int(p.value or 0), int(n.value)


def eng_debug_buffer(e, name: str) -> tuple[int, int]:
    p = ctypes.c_void_p()
    n = ctypes.c_int64()
    _check(e, lib().eng_debug_buffer(e, name.encode(), ctypes.byref(p), ctypes.byref(n)))
    return int(p.value or 0), int(n.value)


def eng_stream(e) -> int:
    return int(lib().eng_stream(e) or 0)


def eng_last_error(e=None) -> str:
    m = lib().eng_last_error(e)
    return m.decode() if m else ""


def eng_destroy(e) -> None:
    lib().eng_destroy(e)


def eng_philox_uniforms(seed: int, offset: int, rows: int, vocab: int, out_dev: int, stream: int | None = None):
    _check(None, lib().eng_philox_uniforms(seed, offset, rows, vocab, out_dev, stream))


def eng_gumbel(u_dev: int, g_dev: int, n: int, stream: int | None = None):
    _check(None, lib().eng_gumbel(u_dev, g_dev, n, stream))


def eng_sample(logits_dev: int, rows: int, vocab: int, temperature, seed: int, offset: int, out_ids_dev: int,
               stream: int | None = None):
    t = np.ascontiguousarray(temperature, dtype=np.float32)
    _check(None, lib().eng_sample(logits_dev, rows, vocab, t.ctypes.data_as(_F32P), seed, offset, out_ids_dev,
                                  stream))


def eng_sample_noalloc(logits_dev: int, rows: int, vocab: int, temperature, seed: int, offset: int,
                       out_ids_dev: int, stream: int | None = None):
    """eng_sample with its per-call scratch in a fixed array of the library (no device allocation)."""
    t = np.ascontiguousarray(temperature, dtype=np.float32)
    _check(None, lib().eng_sample_noalloc(logits_dev, rows, vocab, t.ctypes.data_as(_F32P), seed, offset,
                                          out_ids_dev, stream))


def eng_sample_filtered(logits_dev: int, rows: int, vocab: int, temperature, top_k, top_p, seed: int, offset: int,
                        out_ids_dev: int, out_kept_dev: int | None = None, stream: int | None = None):
    """eng_sample with top-k / top-p filters; top_k or top_p None disables that filter for every row."""
    t = np.ascontiguousarray(temperature, dtype=np.float32)
    k = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32)
    p = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32)
    _check(None, lib().eng_sample_filtered(
        logits_dev, rows, vocab, t.ctypes.data_as(_F32P),
        None if k is None else _ptr_i32(k),
        None if p is None else p.ctypes.data_as(_F32P), seed, offset, out_ids_dev, out_kept_dev, stream))


def eng_exp_f32(d_dev: int, out_dev: int, n: int, stream: int | None = None):
    _check(None, lib().eng_exp_f32(d_dev, out_dev, n, stream))


def eng_generate(e, num_reqs: int, max_steps: int, check_every: int, stop_ids=()):
    """Decode steps with a stop check every check_every steps; returns (tokens [R, max_steps], lengths [R],
    steps run).  Tokens past a request's length are -1."""
    stops = _i32(list(stop_ids))
    toks = np.full((num_reqs, max_steps), -2, dtype=np.int32)
    lens = np.zeros(num_reqs, dtype=np.int32)
    n = _check(e, lib().eng_generate(e, max_steps, check_every, _ptr_i32(stops) if len(stops) else None, len(stops),
                                     _ptr_i32(toks), _ptr_i32(lens)))
    return toks, lens, n


# ------------------------------------------------------------------ mixture of experts (device pointers)


def eng_moe_route(x_dev: int, w_router_dev: int, num_tokens: int, hidden: int, num_experts: int, top_k: int,
                  weights_dev: int, ids_dev: int, stream: int | None = None):
    _check(None, lib().eng_moe_route(x_dev, w_router_dev, num_tokens, hidden, num_experts, top_k, weights_dev,
                                     ids_dev, stream))


def eng_moe_padded_rows(num_tokens: int, top_k: int, num_experts: int, block_m: int) -> int:
    return int(lib().eng_moe_padded_rows(num_tokens, top_k, num_experts, block_m))


def eng_moe_align(ids_dev: int, num_tokens: int, top_k: int, num_experts: int, block_m: int, sorted_ids_dev: int,
                  block_expert_dev: int, info_dev: int, stream: int | None = None):
    _check(None, lib().eng_moe_align(ids_dev, num_tokens, top_k, num_experts, block_m, sorted_ids_dev,
                                     block_expert_dev, info_dev, stream))


def eng_moe_workspace_bytes(num_tokens: int, top_k: int, num_experts: int, hidden: int, inter: int) -> int:
    return int(lib().eng_moe_workspace_bytes(num_tokens, top_k, num_experts, hidden, inter))


def eng_moe_mlp(x_dev: int, gate_up_dev: int, down_dev: int, weights_dev: int, ids_dev: int, num_tokens: int,
                hidden: int, inter: int, num_experts: int, top_k: int, out_dev: int, workspace_dev: int,
                workspace_bytes: int, stream: int | None = None):
    _check(None, lib().eng_moe_mlp(x_dev, gate_up_dev, down_dev, weights_dev, ids_dev, num_tokens, hidden, inter,
                                   num_experts, top_k, out_dev, workspace_dev, workspace_bytes, stream))
