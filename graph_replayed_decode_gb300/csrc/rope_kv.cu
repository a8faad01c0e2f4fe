// rope_kv.cu -- per-head QK-RMSNorm, RoPE, and the paged KV-cache write, in one pass.
//
// "33. Removing overhead", section "Fewer, larger matmuls": RoPE applied inside the KV-write kernel is a
// fusion that saves a pass over memory and a launch without changing the math (stretch exercise 4 asks
// for exactly this kernel).  "19. Fast decode", section "Where the time goes": Qwen3 runs two QK-norms
// per layer.  Section "CUDA graphs for a changing batch" of the first page: a padding row's slot is -1
// and its write lands in a scratch block the block manager never hands out.
//
// One warp per (token, head) of the fused QKV output: q heads are normed (Qwen3), rotated and stored as
// bf16 for attention; k heads are normed, rotated and stored into the paged pool; v heads are stored as
// they are.  The slot of position p of request r is block_tables[r][p / 16] * 16 + p % 16; a row with
// sequence length 0 is padding and writes to the scratch block.  Out-of-range block ids or positions
// are redirected to the scratch block and flagged in the status word (never an out-of-bounds write).
#include "common.cuh"
#include "kernels.h"

namespace grd {

template <int D>
__global__ void __launch_bounds__(256) k_rope_kv(RopeKvParams p) {
  constexpr int E = D / 32;  // values per lane
  pdl_wait();
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.y * 8 + warp;
  const int nheads = p.Hq + 2 * p.Hkv;
  if (head >= nheads) return;

  const int r = p.tok2req[t];
  int pos = p.positions[t];
  const bool padding = p.seq_lens[r] == 0;

  // slot of this token (computed redundantly by every warp; cheap)
  int blk = p.NB, off = 0;
  bool bad = false;
  if (!padding) {
    const int bi = pos >> 4;
    if (pos < 0 || bi >= p.mbs || pos >= p.max_pos) {
      bad = true;
      if (head == 0 && lane == 0) set_status(p.status, ST_BAD_POSITION);
    } else {
      const int b = p.bt[(size_t)r * p.mbs + bi];
      if (b < 0 || b >= p.NB) {
        bad = true;
        if (head == 0 && lane == 0) set_status(p.status, ST_BAD_BLOCK);
      } else {
        blk = b;
        off = pos & 15;
      }
    }
  }
  if (head == 0 && lane == 0) p.slots[t] = (padding || bad) ? -1 : blk * 16 + off;
  if (pos < 0 || pos >= p.max_pos) pos = 0;

  const float* src = p.qkv + (size_t)t * nheads * D + (size_t)head * D + lane * E;
  float x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = src[e];

  const bool is_q = head < p.Hq;
  const bool is_k = !is_q && head < p.Hq + p.Hkv;
  if (is_q || is_k) {
    const float* nw = is_q ? p.q_norm : p.k_norm;
    if (nw) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) ss += x[e] * x[e];
      ss = warp_sum(ss);
      const float rs = rsqrtf(ss / (float)D + p.eps);
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = x[e] * rs * nw[lane * E + e];
    }
    // rotate-half RoPE: element i < D/2 pairs with i + D/2, held by lane ^ 16
    const float* cs = p.cos_sin + (size_t)pos * D;  // [D/2][2]
    float y[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
      const int i = (lane & 15) * E + e;
      const float c = cs[2 * i], sn = cs[2 * i + 1];
      y[e] = (lane < 16) ? (x[e] * c - other * sn) : (x[e] * c + other * sn);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = y[e];
  }

  bf16* dst;
  if (is_q) {
    dst = p.q_out + ((size_t)t * p.Hq + head) * D;
  } else {
    const int kvh = is_k ? head - p.Hq : head - p.Hq - p.Hkv;
    bf16* plane = is_k ? p.k_pool : p.v_pool;
    dst = plane + (((size_t)blk * p.Hkv + kvh) * 16 + off) * D;
  }
  if (E == 4) {
    uint2 v;
    v.x = pack_bf16x2(x[0], x[1]);
    v.y = pack_bf16x2(x[2], x[3]);
    *reinterpret_cast<uint2*>(dst + lane * E) = v;
  } else {
#pragma unroll
    for (int e = 0; e < E; e += 2) *reinterpret_cast<uint32_t*>(dst + lane * E + e) = pack_bf16x2(x[e], x[e + 1]);
  }
  pdl_trigger();
}

cudaError_t launch_rope_kv(const RopeKvParams& p, const LaunchOpts& o, cudaStream_t s) {
  if (p.T <= 0) return cudaSuccess;
  const int nheads = p.Hq + 2 * p.Hkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.T, (nheads + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.d == 128) return cudaLaunchKernelEx(&cfg, k_rope_kv<128>, p);
  if (p.d == 64) return cudaLaunchKernelEx(&cfg, k_rope_kv<64>, p);
  return cudaErrorInvalidValue;
}

}  // namespace grd
