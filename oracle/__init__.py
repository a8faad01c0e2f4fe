"""CPU oracle for the fused serving step -- TEST INFRASTRUCTURE, not a product path.

A plain, slow, obviously correct restatement of what one serving step of a
Qwen3/Qwen2.5-style dense decoder computes, written from the pages:

  * "33. Removing overhead: fusion, graphs and async scheduling"
  * "19. Fast decode: syncs, CUDA graphs and compilation"
  * "One forward per step"
  * "(7) Graph Mode: CUDA Graphs and How vLLM / SGLang Implement Them"

Floating point runs in float64 (the pages fix no activation precision); the
sampler runs in float32 because its float result decides an integer (the
argmax), and that decision is taken in the kernel's precision on both sides.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and never imports it; the only common code is the ``synth`` input generators.

Parity status of each function is stated in its docstring; end-to-end logits
are a composition of pinned parts (no page prints logits for any model).
"""
from .model import (
    OracleModel,
    ContiguousCache,
    PagedCache,
    widen_bf16,
    round_bf16,
    widen_f16,
    round_f16,
    rms_norm,
    silu,
    rope_inv_freq,
    apply_rope,
    attend_one,
    attend_rows,
    attend_packed,
    forward_step,
    fused_qkv,
    fused_gate_up,
)
from .sampler import (
    philox4x32_10,
    uniforms,
    ln_f32,
    gumbel_f32,
    sample,
    sample_row,
)
from .filters import (
    exp_f32,
    sample_filtered,
    sample_row_filtered,
    survivor_counts,
)
from .pool import BlockPool, PoolExhausted, blocks_needed
from .scheduling import gather_input_ids, stop_trim

__all__ = [
    "OracleModel", "ContiguousCache", "PagedCache", "widen_bf16", "round_bf16", "widen_f16", "round_f16", "rms_norm", "silu", "rope_inv_freq",
    "apply_rope", "attend_one", "attend_rows", "attend_packed", "forward_step", "fused_qkv",
    "fused_gate_up", "philox4x32_10", "uniforms", "ln_f32", "gumbel_f32", "sample", "sample_row",
    "exp_f32", "sample_filtered", "sample_row_filtered", "survivor_counts",
    "BlockPool", "PoolExhausted", "blocks_needed", "gather_input_ids", "stop_trim",
]
