"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark.

This package holds model shapes and deterministic input generators only: weights,
prompts, context lengths and pre-filled KV contents.  It contains none of the
decoder's arithmetic (no norm, projection, attention or sampling), so the CPU
oracle and the CUDA path can both consume its outputs without sharing code.
"""
from .configs import CONFIGS, MOE_CONFIGS, ModelShape, MoeShape, moe_shape, shape
from .inputs import (
    Streams,
    bf16_bits_from_f32,
    f32_from_bf16_bits,
    normal_bf16,
    normal_f16,
    make_weights,
    weight_names,
    prompt_ids,
    decode_ids,
    context_lengths,
    kv_context,
    mixed_chunk_prompts,
    moe_weights,
    moe_tokens,
)

__all__ = [
    "CONFIGS", "ModelShape", "shape", "Streams", "bf16_bits_from_f32", "f32_from_bf16_bits",
    "normal_bf16", "normal_f16", "make_weights", "weight_names", "prompt_ids", "decode_ids", "context_lengths", "kv_context",
    "mixed_chunk_prompts", "MOE_CONFIGS", "MoeShape", "moe_shape", "moe_weights", "moe_tokens",
]
