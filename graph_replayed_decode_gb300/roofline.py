"""Algorithmic byte and FLOP counts of one serving step (pure Python, no GPU needed).

"19. Fast decode", §Where the time goes: the decode ceiling is the weight bytes
read per token divided by the memory bandwidth (1.19 GB for Qwen3-0.6B in BF16
at 1,008 GB/s gives about 840 tokens/s).  "One forward per step", §Bottleneck:
the pure-decode step spends 5.15 ms reading Qwen2.5-1.5B's weights on the A10.
The step roofline here extends that count with the KV cache traffic:

  bytes = every layer weight + final norm + LM head, read once
        + the gathered embedding rows (T x hidden)
        + KV read: for each request, seq_len x 2 x kv_heads x head_dim x 2 B per layer
        + KV written: T x 2 x kv_heads x head_dim x 2 B per layer
  flops = 2 T (layer parameters) + 2 R vocab hidden + 4 q_heads head_dim (keys seen by all queries) per layer

Padding rows and activations (well under 1 % at these shapes) are left out.
"""
from __future__ import annotations

from typing import Sequence


def layer_params(s) -> int:
    n = s.hidden * s.qkv_size + s.q_size * s.hidden + 3 * s.intermediate * s.hidden + 2 * s.hidden
    if s.qkv_bias:
        n += s.qkv_size
    if s.qk_norm:
        n += 2 * s.head_dim
    return n


def weight_params(s) -> int:
    """Parameters read by one step: all layers, the final norm and the LM head (once)."""
    return s.layers * layer_params(s) + s.hidden + s.vocab * s.hidden


def weight_bytes(s, elem: int = 2) -> int:
    return weight_params(s) * elem


def kv_bytes_per_token(s, elem: int = 2) -> int:
    """K and V of one position across all layers."""
    return s.layers * 2 * s.kv_heads * s.head_dim * elem


def step_bytes(s, num_tokens: int, seq_lens: Sequence[int], elem: int = 2) -> int:
    """Algorithmic HBM bytes of one step with ``num_tokens`` packed tokens.

    ``seq_lens[r]`` is the number of keys request r's last query sees; a request
    with a multi-token chunk reads its keys once, like a decode row.
    """
    b = weight_bytes(s, elem)
    b += num_tokens * s.hidden * elem
    b += sum(int(x) for x in seq_lens) * kv_bytes_per_token(s, elem)
    b += num_tokens * kv_bytes_per_token(s, elem)
    return b


def step_flops(s, num_tokens: int, num_reqs: int, keys_seen: int) -> int:
    """FLOPs of one step; ``keys_seen`` = keys summed over all packed queries."""
    f = 2 * num_tokens * s.layers * layer_params(s)
    f += 2 * num_reqs * s.vocab * s.hidden
    f += 4 * s.q_heads * s.head_dim * keys_seen * s.layers
    return f


def decode_ceiling_tokens_per_s(s, bandwidth_bytes_per_s: float, elem: int = 2) -> float:
    """Batch-1 ceiling of "19. Fast decode": weight bytes per token over bandwidth."""
    return bandwidth_bytes_per_s / weight_bytes(s, elem)


def roofline_seconds(bytes_: float, flops: float, bandwidth: float, peak_flops: float) -> float:
    return max(bytes_ / bandwidth, flops / peak_flops)
