"""Reference forward of one packed serving step, in float64 -- TEST INFRASTRUCTURE.

One step takes an unpadded packed sequence (prefill chunks first, decode tokens
last; "One forward per step", §What changed) and returns, for every request,
the logits at its last packed token ("33. Removing overhead", §CUDA graphs for
a changing batch: one logits row per request).

The decoder is the plain Qwen-style stack the pages enumerate ("19. Fast
decode", §Where the time goes): per layer an RMSNorm, the Q/K/V projections,
per-head QK-norms, RoPE on Q and K, the cache write, attention, the output
projection and a residual add, a second RMSNorm, the gate and up projections,
SiLU, the product, the down projection and a second residual add.  The oracle
keeps the projections separate (unfused) and computes in float64 from the
exact float64 widening of the bf16 weights.

Readings where the pages are silent:
  * RMSNorm: x / sqrt(mean(x^2) + eps) * w.
  * QK-norm: the same RMSNorm over each head's head_dim values with one shared
    [head_dim] weight, applied before RoPE; absent on QKV-bias models.
  * RoPE: rotate-half convention, inv_freq_i = theta^(-2i/d), angle = pos * inv_freq_i.
  * attention: scale 1/sqrt(d); a query at position p sees keys 0..p of its own
    request; query head h reads KV head h // (q_heads / kv_heads); a row whose
    sequence length is 0 (a padding row) outputs zeros.
"""
from __future__ import annotations

import numpy as np

from synth import ModelShape

# ----------------------------------------------------------------------------- elementwise pieces


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns as float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even (8 significant bits).

    Written from the format's definition: x = m * 2^e with 0.5 <= |m| < 1, so m * 2^8 rounded to an
    integer (numpy's rint rounds half to even) is the 8-bit significand.  Finite values inside bf16's
    normal range only.  Pinned against torch's float32 -> bfloat16 conversion and against brute-force
    nearest-neighbour rounding.
    """
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def widen_f16(bits: np.ndarray) -> np.ndarray:
    """Exact value of IEEE binary16 bit patterns as float64, from the format's definition.

    Sign bit 15, exponent bits 14..10 (bias 15), 10 fraction bits: a normal number is
    (1 + f/1024) * 2^(e - 15), a subnormal (e = 0) is f/1024 * 2^-14, e = 31 is inf (f = 0) or NaN.
    Pinned against numpy's half-precision type on all 65,536 patterns.
    """
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 10) & 31
    f = (b & 1023).astype(np.float64)
    normal = np.ldexp(1.0 + f / 1024.0, (e - 15).astype(np.int32))
    sub = np.ldexp(f / 1024.0, -14)
    special = np.where(f == 0, np.inf, np.nan)
    return sign * np.where(e == 0, sub, np.where(e == 31, special, normal))


F16_MAX = 65504.0


def round_f16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest IEEE binary16 value, ties to even.

    From the format's definition: at and above 2^-14 a value has 11 significant bits, so with
    x = m * 2^e (0.5 <= |m| < 1) the significand is rint(m * 2^11) (numpy's rint rounds half to
    even); below 2^-14 the spacing is the fixed 2^-24 of the subnormals.  Results past the largest
    finite value (65504) are infinite.  Pinned against numpy's float64 -> float16 conversion.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    normal = np.ldexp(np.rint(np.ldexp(m, 11)), e - 11)
    sub = np.ldexp(np.rint(np.ldexp(x, 24)), -24)
    r = np.where(np.abs(x) >= 2.0 ** -14, normal, sub)
    return np.where(np.abs(r) > F16_MAX, np.copysign(np.inf, x), r)


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis.

    "33. Removing overhead", §Fewer, larger matmuls (add_norm: a layer's
    residual add followed by the next norm); the formula itself is not printed
    on the pages, so the standard definition is used.  Pinned by the library
    routine torch.nn.functional.rms_norm and by the constant-vector closed form.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g / (1 + e^-g): "33. Removing overhead", silu_and_mul kernel.  Pinned by torch silu."""
    return g / (1.0 + np.exp(-g))


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * i / head_dim)


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotary embedding, rotate-half form, on x [n, heads, d] at absolute positions [n].

    "33. Removing overhead" names RoPE applied inside the KV-write kernel as a
    fusion that does not change the math; the rotation convention is not
    printed, so the rotate-half (NeoX / Qwen) form is taken.  Pinned by the
    closed forms: identity at position 0, norm preservation, relative-position
    dependence of <R_m q, R_n k>, and complex multiplication when d = 2.
    """
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(d, theta)[None, :]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def fused_qkv(wq: np.ndarray, wk: np.ndarray, wv: np.ndarray) -> np.ndarray:
    """[W_Q | W_K | W_V] stacked along the output axis ("33. Removing overhead", §Fewer, larger matmuls)."""
    return np.concatenate([wq, wk, wv], axis=0)


def fused_gate_up(wg: np.ndarray, wu: np.ndarray) -> np.ndarray:
    """[W_gate | W_up] stacked along the output axis ("33. Removing overhead", §Fewer, larger matmuls)."""
    return np.concatenate([wg, wu], axis=0)


# ----------------------------------------------------------------------------- KV caches


class ContiguousCache:
    """Per-request cache indexed by absolute position, zero-filled, full capacity on read.

    "19. Fast decode", §Static shapes and a static cache: keys are written at
    their absolute positions in a preallocated zero buffer, reads return the
    whole capacity with key positions 0..capacity-1, and the causal rule
    key_pos <= query_pos hides slots that were never written.
    """

    def __init__(self, s: ModelShape, capacity: dict[int, int]):
        self.s = s
        self.capacity = dict(capacity)
        self.keys = {(l, r): np.zeros((s.kv_heads, cap, s.head_dim)) for r, cap in capacity.items()
                     for l in range(s.layers)}
        self.values = {(l, r): np.zeros((s.kv_heads, cap, s.head_dim)) for r, cap in capacity.items()
                       for l in range(s.layers)}

    def write(self, layer: int, r: int, positions, k: np.ndarray, v: np.ndarray) -> None:
        positions = np.asarray(positions)
        if positions.size and int(positions.max()) >= self.capacity[r]:
            raise ValueError("position exceeds the cache capacity")
        self.keys[(layer, r)][:, positions, :] = np.swapaxes(k, 0, 1)
        self.values[(layer, r)][:, positions, :] = np.swapaxes(v, 0, 1)

    def read(self, layer: int, r: int, n_keys: int):
        """All ``capacity`` slots and their positions (the causal rule masks the rest)."""
        cap = self.capacity[r]
        return self.keys[(layer, r)], self.values[(layer, r)], np.arange(cap)


class PagedCache:
    """Paged pool of fixed-size blocks reached through per-request block tables.

    "33. Removing overhead", §CUDA graphs for a changing batch: each token has a
    slot; slot -1 (a padding row) is redirected to a scratch block that the
    block manager never hands out.  "One forward per step": the KV pool is made
    of fixed-size blocks.  The slot of position p of request r is
    block_table[r][p // block_size] * block_size + p % block_size.
    Blocks are stored sparsely (only those written) so that a large pool costs
    nothing until used.
    """

    def __init__(self, s: ModelShape, num_blocks: int, block_size: int = 16):
        self.s = s
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.scratch = num_blocks
        self.block_tables: dict[int, list[int]] = {}
        self._blocks: dict[tuple[int, int], np.ndarray] = {}

    def set_block_table(self, r: int, blocks) -> None:
        self.block_tables[r] = [int(b) for b in blocks]

    def slot(self, r: int | None, pos: int) -> int:
        if r is None:
            return -1
        table = self.block_tables[r]
        b = pos // self.block_size
        if b >= len(table):
            raise ValueError("position exceeds the request's block table")
        return table[b] * self.block_size + pos % self.block_size

    def _block(self, layer: int, blk: int) -> np.ndarray:
        key = (layer, blk)
        if key not in self._blocks:
            self._blocks[key] = np.zeros((2, self.s.kv_heads, self.block_size, self.s.head_dim))
        return self._blocks[key]

    def write_slot(self, layer: int, slot: int, k: np.ndarray, v: np.ndarray) -> None:
        if slot < 0:
            blk, off = self.scratch, 0
        else:
            blk, off = divmod(slot, self.block_size)
        b = self._block(layer, blk)
        b[0, :, off, :] = k
        b[1, :, off, :] = v

    def write(self, layer: int, r: int, positions, k: np.ndarray, v: np.ndarray) -> None:
        for i, p in enumerate(np.asarray(positions)):
            self.write_slot(layer, self.slot(r, int(p)), k[i], v[i])

    def read(self, layer: int, r: int, n_keys: int):
        """Keys and values of positions 0..n_keys-1 gathered through the block table."""
        K = np.zeros((self.s.kv_heads, n_keys, self.s.head_dim))
        V = np.zeros((self.s.kv_heads, n_keys, self.s.head_dim))
        for p0 in range(0, n_keys, self.block_size):
            blk = self.block_tables[r][p0 // self.block_size]
            b = self._block(layer, blk)
            n = min(self.block_size, n_keys - p0)
            K[:, p0:p0 + n, :] = b[0, :, :n, :]
            V[:, p0:p0 + n, :] = b[1, :, :n, :]
        return K, V, np.arange(n_keys)

    def block_contents(self, layer: int, blk: int) -> np.ndarray:
        return self._block(layer, blk)


# ----------------------------------------------------------------------------- attention


def attend_one(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q K^T * scale) V for one query vector q [d] over keys K, V [n, d]."""
    if K.shape[0] == 0:
        return np.zeros_like(q)
    s = (K @ q) * scale
    s = s - s.max()
    p = np.exp(s)
    return (p / p.sum()) @ V


def attend_rows(s: ModelShape, cache, layer: int, q: np.ndarray, reqs, positions) -> np.ndarray:
    """One query row per request: the decode-side kernel of the split.

    "One forward per step", §What changed: decode positions are reshaped to one
    query row per request and each row reads only its own request's history.
    q [n, q_heads, d]; reqs[i] is the request of row i (None for a padding row,
    which outputs zeros); positions[i] its absolute position.
    """
    group = s.q_heads // s.kv_heads
    scale = 1.0 / np.sqrt(s.head_dim)
    out = np.zeros_like(q)
    for i, (r, p) in enumerate(zip(reqs, positions)):
        if r is None:
            continue
        K, V, kpos = cache.read(layer, r, int(p) + 1)
        vis = kpos <= int(p)
        for h in range(s.q_heads):
            g = h // group
            out[i, h] = attend_one(q[i, h], K[g][vis], V[g][vis], scale)
    return out


def attend_packed(s: ModelShape, cache, layer: int, q: np.ndarray, r: int, positions) -> np.ndarray:
    """Causal attention for one request's packed chunk as a single masked matrix product.

    "One forward per step", §What changed: chunk positions run a packed causal
    prefill kernel.  q [n, q_heads, d] holds the chunk's queries at absolute
    positions [n]; keys 0..max(positions) come from the cache (earlier chunks
    and this chunk, already written), masked by key_pos <= query_pos.
    """
    positions = np.asarray(positions)
    group = s.q_heads // s.kv_heads
    scale = 1.0 / np.sqrt(s.head_dim)
    K, V, kpos = cache.read(layer, r, int(positions.max()) + 1)
    mask = kpos[None, :] <= positions[:, None]                      # [n, keys]
    out = np.zeros_like(q)
    for h in range(s.q_heads):
        g = h // group
        sc = (q[:, h, :] @ K[g].T) * scale                           # [n, keys]
        sc = np.where(mask, sc, -np.inf)
        sc = sc - sc.max(axis=1, keepdims=True)
        p = np.exp(sc)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ V[g]
    return out


# ----------------------------------------------------------------------------- model


class OracleModel:
    """Float64 view of bf16 (or fp16) weights given by Hugging Face tensor name.

    ``weights`` maps a name to a uint16 bit array (for example the lazy
    ``synth`` generator); ``dtype`` names the 16-bit format of those bits
    ("bf16" or "f16").  Widened tensors are cached per layer when
    ``cache_layers`` is true; otherwise they are widened on every use, which
    keeps the memory of large shapes bounded.
    """

    def __init__(self, s: ModelShape, weights, cache_layers: bool = True, dtype: str = "bf16"):
        if dtype not in ("bf16", "f16"):
            raise ValueError(f"dtype must be 'bf16' or 'f16', not {dtype!r}")
        self.s = s
        self.w = weights
        self.cache_layers = cache_layers
        self.dtype = dtype
        self._widen = widen_bf16 if dtype == "bf16" else widen_f16
        self._memo: dict[str, np.ndarray] = {}

    def get(self, name: str) -> np.ndarray:
        if name in self._memo:
            return self._memo[name]
        a = self._widen(self.w[name])
        if self.cache_layers:
            self._memo[name] = a
        return a

    def has(self, name: str) -> bool:
        return name in self.w

    def embed(self) -> np.ndarray:
        return self.get("model.embed_tokens.weight")

    def lm_head(self) -> np.ndarray:
        if self.s.tie_embeddings:
            return self.embed()
        return self.get("lm_head.weight")


def _requests_of_tokens(cu_seqlens: np.ndarray) -> np.ndarray:
    T = int(cu_seqlens[-1])
    req = np.zeros(T, dtype=np.int64)
    for r in range(len(cu_seqlens) - 1):
        req[cu_seqlens[r]:cu_seqlens[r + 1]] = r
    return req


def forward_step(model: OracleModel, cache, token_ids, positions, cu_seqlens, request_keys=None,
                 attention: str = "split", return_hidden: bool = False, activations: str = "f64"):
    """Run one packed step and return logits [R, vocab] at each request's last token.

    token_ids, positions: [T]; cu_seqlens: [R + 1] (request r owns tokens
    cu_seqlens[r] .. cu_seqlens[r+1]-1, prefill chunks first, decode tokens last).
    ``request_keys[r]`` names request r in ``cache`` (default r).

    attention="split" runs leading multi-token requests through the packed causal
    routine and single-token requests through the row routine ("One forward per
    step", §What changed); "rows" sends every token through the row routine and
    "packed" every request through the packed routine.  All three compute the
    same values; the tests pin them against each other.

    activations="f64" keeps every activation in float64.  activations="bf16" is the
    precision the parity bar is stated for: a BF16 model ("19. Fast decode") whose
    kernels compute in fp32 and store their outputs in the activation type ("33.
    Removing overhead", silu_and_mul).  Every operand a contraction reads is
    rounded to bf16 -- the normed inputs of the QKV, gate|up and LM-head
    projections, Q and the cached K/V (after QK-norm and RoPE), the attention
    output, the SiLU-and-mul product -- while the sums themselves (the
    projections, the attention softmax and weighted sum, the residual stream that
    accumulates every layer's output) stay in float64.  The QK-norm, RoPE and
    SiLU-and-mul act on the unrounded projection sums, as they do when fused into
    the projection that produces them.  activations="f16" is the same with IEEE
    binary16 in place of bf16 (the fp16 variant of a model).
    """
    if activations not in ("f64", "bf16", "f16"):
        raise ValueError(f"activations must be 'f64', 'bf16' or 'f16', not {activations!r}")
    act = {"bf16": round_bf16, "f16": round_f16}.get(activations, lambda a: a)
    s = model.s
    token_ids = np.asarray(token_ids, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    R = len(cu) - 1
    keys = list(range(R)) if request_keys is None else list(request_keys)
    req_of = _requests_of_tokens(cu)
    tok_key = [keys[r] for r in req_of]
    qlen = np.diff(cu)

    h = model.embed()[token_ids].copy()
    for l in range(s.layers):
        p = f"model.layers.{l}."
        x = act(rms_norm(h, model.get(p + "input_layernorm.weight"), s.rms_eps))
        q = x @ model.get(p + "self_attn.q_proj.weight").T
        k = x @ model.get(p + "self_attn.k_proj.weight").T
        v = x @ model.get(p + "self_attn.v_proj.weight").T
        if s.qkv_bias:
            q = q + model.get(p + "self_attn.q_proj.bias")
            k = k + model.get(p + "self_attn.k_proj.bias")
            v = v + model.get(p + "self_attn.v_proj.bias")
        T = len(token_ids)
        q = q.reshape(T, s.q_heads, s.head_dim)
        k = k.reshape(T, s.kv_heads, s.head_dim)
        v = v.reshape(T, s.kv_heads, s.head_dim)
        if s.qk_norm:
            q = rms_norm(q, model.get(p + "self_attn.q_norm.weight"), s.rms_eps)
            k = rms_norm(k, model.get(p + "self_attn.k_norm.weight"), s.rms_eps)
        q = apply_rope(q, positions, s.rope_theta)
        k = apply_rope(k, positions, s.rope_theta)
        q, k, v = act(q), act(k), act(v)
        for r in range(R):
            sl = slice(cu[r], cu[r + 1])
            cache.write(l, keys[r], positions[sl], k[sl], v[sl])

        o = np.zeros_like(q)
        if attention == "rows":
            o[:] = attend_rows(s, cache, l, q, tok_key, positions)
        else:
            n_packed = R
            if attention == "split":
                n_packed = 0
                for r in range(R):
                    if qlen[r] > 1:
                        n_packed = r + 1
            for r in range(n_packed):
                sl = slice(cu[r], cu[r + 1])
                if cu[r + 1] > cu[r]:
                    o[sl] = attend_packed(s, cache, l, q[sl], keys[r], positions[sl])
            if n_packed < R:
                sl = slice(cu[n_packed], cu[R])
                o[sl] = attend_rows(s, cache, l, q[sl], tok_key[cu[n_packed]:], positions[sl])
        h = h + act(o.reshape(T, s.q_size)) @ model.get(p + "self_attn.o_proj.weight").T
        x = act(rms_norm(h, model.get(p + "post_attention_layernorm.weight"), s.rms_eps))
        g = x @ model.get(p + "mlp.gate_proj.weight").T
        u = x @ model.get(p + "mlp.up_proj.weight").T
        h = h + act(silu(g) * u) @ model.get(p + "mlp.down_proj.weight").T

    last = cu[1:] - 1
    y = act(rms_norm(h[last], model.get("model.norm.weight"), s.rms_eps))
    logits = y @ model.lm_head().T
    if return_hidden:
        return logits, h
    return logits
