"""Model shapes of the five decoder workloads (dimensions only, no arithmetic).

The shapes follow the workloads the pages measure: a Qwen3-0.6B-shaped decoder
("19. Fast decode", §Where the time goes: 28 layers, BF16), a Qwen2.5-1.5B-shaped
decoder ("One forward per step", setup paragraph of §What changed), an 8B-shaped
dense decoder and a tiny two-layer test model.  Values the pages leave open are
fixed here: eps 1e-6, RoPE theta 1e6, QK-norm on
the Qwen3-style shapes (tiny, 0.6B, 8B), QKV bias on the Qwen2.5 shape, tied
embeddings everywhere except the 8B shape.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict


@dataclass(frozen=True)
class ModelShape:
    name: str
    layers: int
    hidden: int
    q_heads: int
    kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    qk_norm: bool = True
    qkv_bias: bool = False
    tie_embeddings: bool = True

    @property
    def q_size(self) -> int:
        return self.q_heads * self.head_dim

    @property
    def kv_size(self) -> int:
        return self.kv_heads * self.head_dim

    @property
    def qkv_size(self) -> int:
        return self.q_size + 2 * self.kv_size

    def as_dict(self) -> dict:
        return asdict(self)


CONFIGS = {
    "tiny": ModelShape("tiny", layers=2, hidden=256, q_heads=4, kv_heads=2, head_dim=64,
                       intermediate=768, vocab=4096, qk_norm=True, qkv_bias=False, tie_embeddings=True),
    "qwen3_0p6b": ModelShape("qwen3_0p6b", layers=28, hidden=1024, q_heads=16, kv_heads=8, head_dim=128,
                             intermediate=3072, vocab=151936, qk_norm=True, qkv_bias=False,
                             tie_embeddings=True),
    "qwen2p5_1p5b": ModelShape("qwen2p5_1p5b", layers=28, hidden=1536, q_heads=12, kv_heads=2, head_dim=128,
                               intermediate=8960, vocab=151936, qk_norm=False, qkv_bias=True,
                               tie_embeddings=True),
    "dense_8b": ModelShape("dense_8b", layers=36, hidden=4096, q_heads=32, kv_heads=8, head_dim=128,
                           intermediate=12288, vocab=151936, qk_norm=True, qkv_bias=False,
                           tie_embeddings=False),
}


def shape(name: str) -> ModelShape:
    return CONFIGS[name]


@dataclass(frozen=True)
class MoeShape:
    """One mixture-of-experts MLP: E experts of SwiGLU width `intermediate`, k experts per token."""
    name: str
    hidden: int
    experts: int
    top_k: int
    intermediate: int

    def as_dict(self) -> dict:
        return asdict(self)


# The pages name Qwen3-30B-A3B (128 experts); its published layer widths are hidden 2048, 8 experts per token
# and expert width 768.  The tiny shape is for the oracle's own tests.
MOE_CONFIGS = {
    "tiny_moe": MoeShape("tiny_moe", hidden=64, experts=8, top_k=2, intermediate=32),
    "qwen3_30b_a3b_moe": MoeShape("qwen3_30b_a3b_moe", hidden=2048, experts=128, top_k=8, intermediate=768),
}


def moe_shape(name: str) -> MoeShape:
    return MOE_CONFIGS[name]
