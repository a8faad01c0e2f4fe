"""Deterministic synthetic inputs: weights, prompts, context lengths and KV contents.

Every generator draws from ``numpy.random.default_rng([seed, stream, ...])`` so
that each purpose (weights, prompts, context lengths, KV fill, chunk mix) has
its own stream and any single tensor can be regenerated without the others.

Recipe (the pages run real checkpoints; these stand in for them):
  * matrices and biases ~ N(0, 0.02), bf16: a 16-bit uniform integer indexes a
    table of bf16-rounded normal quantiles at (k + 0.5) / 65536, so the values
    follow N(0, 0.02) truncated at about 4.3 sigma, at a cost of one table
    lookup per weight; with dtype "f16" the same integers index a table of
    fp16-rounded quantiles (the fp16 variant of a shape: the same draws,
    rounded to the other 16-bit format);
  * RMSNorm and QK-norm weights = 1.0 (N(0, 0.02) norm weights would drive
    every activation towards zero); with ``norm_scale`` > 0 they are instead
    bf16 draws of 1 + N(0, norm_scale^2) from the tensor's own stream (the same
    quantile-table method), so that every norm weight differs from its
    neighbours and from the other norms' weights;
  * prompt ids uniform over the vocabulary;
  * pre-filled context K/V ~ N(0, 1), bf16, by the same table method.
"""
from __future__ import annotations

import functools
from typing import Iterator

import numpy as np
from scipy.special import ndtri

from .configs import ModelShape, MoeShape


class Streams:
    WEIGHTS = 1
    PROMPTS = 2
    CONTEXTS = 3
    KV = 4
    CHUNK = 5
    DECODE_IDS = 6
    MOE = 7


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); returns uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@functools.lru_cache(maxsize=8)
def _quantile_table(scale: float) -> np.ndarray:
    k = np.arange(65536, dtype=np.float64)
    q = ndtri((k + 0.5) / 65536.0) * scale
    return bf16_bits_from_f32(q.astype(np.float32))


@functools.lru_cache(maxsize=8)
def _quantile_table_shifted(scale: float, shift: float) -> np.ndarray:
    k = np.arange(65536, dtype=np.float64)
    q = shift + ndtri((k + 0.5) / 65536.0) * scale
    return bf16_bits_from_f32(q.astype(np.float32))


@functools.lru_cache(maxsize=8)
def _quantile_table_f16_shifted(scale: float, shift: float) -> np.ndarray:
    k = np.arange(65536, dtype=np.float64)
    q = shift + ndtri((k + 0.5) / 65536.0) * scale
    return q.astype(np.float16).view(np.uint16)


@functools.lru_cache(maxsize=8)
def _quantile_table_f16(scale: float) -> np.ndarray:
    k = np.arange(65536, dtype=np.float64)
    q = ndtri((k + 0.5) / 65536.0) * scale
    return q.astype(np.float16).view(np.uint16)


def _table_indices(rng: np.random.Generator, n: int) -> np.ndarray:
    words = rng.integers(0, 2 ** 32, size=(n + 1) // 2, dtype=np.uint32)
    return words.view(np.uint16)[:n]


def normal_bf16(rng: np.random.Generator, n: int, scale: float) -> np.ndarray:
    """n bf16 values ~ N(0, scale^2) (16-bit quantile table), as uint16 bits."""
    return _quantile_table(float(scale))[_table_indices(rng, n)]


def normal_f16(rng: np.random.Generator, n: int, scale: float) -> np.ndarray:
    """n IEEE fp16 values ~ N(0, scale^2) from the same draws as normal_bf16, as uint16 bits."""
    return _quantile_table_f16(float(scale))[_table_indices(rng, n)]


def _normal(dtype: str):
    if dtype == "bf16":
        return normal_bf16
    if dtype == "f16":
        return normal_f16
    raise ValueError(f"dtype must be 'bf16' or 'f16', not {dtype!r}")


BF16_ONE = np.uint16(0x3F80)
F16_ONE = np.uint16(0x3C00)


def weight_names(s: ModelShape) -> list[tuple[str, tuple[int, ...]]]:
    """Tensor names (Hugging Face Qwen naming) and shapes, in a fixed order."""
    out: list[tuple[str, tuple[int, ...]]] = [("model.embed_tokens.weight", (s.vocab, s.hidden))]
    for i in range(s.layers):
        p = f"model.layers.{i}."
        out.append((p + "input_layernorm.weight", (s.hidden,)))
        out.append((p + "self_attn.q_proj.weight", (s.q_size, s.hidden)))
        out.append((p + "self_attn.k_proj.weight", (s.kv_size, s.hidden)))
        out.append((p + "self_attn.v_proj.weight", (s.kv_size, s.hidden)))
        if s.qkv_bias:
            out.append((p + "self_attn.q_proj.bias", (s.q_size,)))
            out.append((p + "self_attn.k_proj.bias", (s.kv_size,)))
            out.append((p + "self_attn.v_proj.bias", (s.kv_size,)))
        if s.qk_norm:
            out.append((p + "self_attn.q_norm.weight", (s.head_dim,)))
            out.append((p + "self_attn.k_norm.weight", (s.head_dim,)))
        out.append((p + "self_attn.o_proj.weight", (s.hidden, s.q_size)))
        out.append((p + "post_attention_layernorm.weight", (s.hidden,)))
        out.append((p + "mlp.gate_proj.weight", (s.intermediate, s.hidden)))
        out.append((p + "mlp.up_proj.weight", (s.intermediate, s.hidden)))
        out.append((p + "mlp.down_proj.weight", (s.hidden, s.intermediate)))
    out.append(("model.norm.weight", (s.hidden,)))
    if not s.tie_embeddings:
        out.append(("lm_head.weight", (s.vocab, s.hidden)))
    return out


class Weights:
    """Lazily generated bf16 (or fp16) weights, uint16 bit arrays keyed by tensor name.

    Tensor ``i`` of ``weight_names`` is drawn from stream ``[seed, WEIGHTS, i]``,
    so any tensor can be produced alone and in any order with the same bits.
    Norm weights are 1.0, or with ``norm_scale`` > 0 draws of 1 + N(0, norm_scale^2).
    """

    def __init__(self, s: ModelShape, seed: int = 0, cache: bool = True, dtype: str = "bf16",
                 norm_scale: float = 0.0):
        if not norm_scale >= 0.0:
            raise ValueError("norm_scale must be >= 0")
        self.shape = s
        self.seed = seed
        self.dtype = dtype
        self.norm_scale = float(norm_scale)
        self._draw = _normal(dtype)
        self._one = BF16_ONE if dtype == "bf16" else F16_ONE
        self._spec = weight_names(s)
        self._index = {name: i for i, (name, _) in enumerate(self._spec)}
        self._cache: dict[str, np.ndarray] | None = {} if cache else None

    def names(self) -> list[str]:
        return [n for n, _ in self._spec]

    def dims(self, name: str) -> tuple[int, ...]:
        return self._spec[self._index[name]][1]

    def __contains__(self, name: str) -> bool:
        return name in self._index

    def __getitem__(self, name: str) -> np.ndarray:
        if self._cache is not None and name in self._cache:
            return self._cache[name]
        i = self._index[name]
        dims = self._spec[i][1]
        n = int(np.prod(dims))
        if name.endswith("norm.weight") or name.endswith("layernorm.weight"):
            if self.norm_scale == 0.0:
                arr = np.full(dims, self._one, dtype=np.uint16)
            else:
                rng = np.random.default_rng([self.seed, Streams.WEIGHTS, i])
                table = (_quantile_table_shifted if self.dtype == "bf16" else _quantile_table_f16_shifted)(
                    self.norm_scale, 1.0)
                arr = table[_table_indices(rng, n)].reshape(dims)
        else:
            rng = np.random.default_rng([self.seed, Streams.WEIGHTS, i])
            arr = self._draw(rng, n, 0.02).reshape(dims)
        if self._cache is not None:
            self._cache[name] = arr
        return arr

    def items(self) -> Iterator[tuple[str, np.ndarray]]:
        for name in self.names():
            yield name, self[name]

    def drop(self, name: str) -> None:
        if self._cache is not None:
            self._cache.pop(name, None)


def make_weights(s: ModelShape, seed: int = 0, cache: bool = True, dtype: str = "bf16",
                 norm_scale: float = 0.0) -> Weights:
    return Weights(s, seed, cache, dtype, norm_scale)


def prompt_ids(n: int, vocab: int, key: int, seed: int = 0) -> np.ndarray:
    """n token ids uniform on [0, vocab) from stream [seed, PROMPTS, key]."""
    rng = np.random.default_rng([seed, Streams.PROMPTS, key])
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def decode_ids(n: int, vocab: int, key: int, seed: int = 0) -> np.ndarray:
    """Input ids for decode rows whose context is pre-filled synthetically."""
    rng = np.random.default_rng([seed, Streams.DECODE_IDS, key])
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def context_lengths(n: int, choices, key: int = 0, seed: int = 0) -> np.ndarray:
    """n context lengths drawn uniformly from ``choices`` (stream [seed, CONTEXTS, key])."""
    rng = np.random.default_rng([seed, Streams.CONTEXTS, key])
    c = np.asarray(list(choices), dtype=np.int64)
    return c[rng.integers(0, len(c), size=n)].astype(np.int32)


def kv_context(s: ModelShape, layer: int, request_key: int, ctx: int, seed: int = 0,
               dtype: str = "bf16") -> np.ndarray:
    """Synthetic cached K and V for one request and layer: uint16 bf16 (or fp16) bits [2, kv_heads, ctx, head_dim].

    Position p of request ``request_key`` holds the same values whatever the
    block layout, so a paged pool and a contiguous cache can be filled alike.
    """
    rng = np.random.default_rng([seed, Streams.KV, layer, request_key])
    n = 2 * s.kv_heads * ctx * s.head_dim
    return _normal(dtype)(rng, n, 1.0).reshape(2, s.kv_heads, ctx, s.head_dim)


def mixed_chunk_prompts(budget: int = 512, choices=(16, 64, 256, 1024, 4096), key: int = 0,
                        seed: int = 0) -> list[tuple[int, int]]:
    """Fresh prompts admitted first-come-first-served into one chunk of ``budget`` positions.

    Returns (prompt_length, chunk_length) per admitted prompt; the last prompt is
    cut where the budget runs out (its chunk is not final, so it is not sampled).
    """
    rng = np.random.default_rng([seed, Streams.CHUNK, key])
    c = np.asarray(list(choices), dtype=np.int64)
    out: list[tuple[int, int]] = []
    left = budget
    while left > 0:
        plen = int(c[rng.integers(0, len(c))])
        take = min(plen, left)
        out.append((plen, take))
        left -= take
    return out


def moe_weights(m: MoeShape, seed: int = 0, dtype: str = "bf16") -> dict[str, np.ndarray]:
    """One MoE layer's weights as 16-bit patterns: the router [E, D], the experts' gate|up [E, 2I, D]
    (gate rows first, then up rows) and down [E, D, I], all ~ N(0, 0.02), one stream per tensor."""
    draw = _normal(dtype)
    dims = {"router": (m.experts, m.hidden), "gate_up": (m.experts, 2 * m.intermediate, m.hidden),
            "down": (m.experts, m.hidden, m.intermediate)}
    out = {}
    for i, (name, d) in enumerate(dims.items()):
        rng = np.random.default_rng([seed, Streams.MOE, i])
        out[name] = draw(rng, int(np.prod(d)), 0.02).reshape(d)
    return out


def moe_tokens(n: int, hidden: int, key: int = 0, seed: int = 0, dtype: str = "bf16") -> np.ndarray:
    """n normed token rows entering a MoE layer, ~ N(0, 1), as 16-bit patterns [n, hidden]."""
    rng = np.random.default_rng([seed, Streams.MOE, 100 + key])
    return _normal(dtype)(rng, n * hidden, 1.0).reshape(n, hidden)
