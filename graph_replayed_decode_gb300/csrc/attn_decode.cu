// attn_decode.cu -- paged decode attention: one query row per request, split over the key length.
//
// "One forward per step", section "What changed": decode positions are reshaped to one query row per
// request so that every request's history is read in parallel (0.347 ms as rows vs 1.749 ms packed on
// the page's A10), and section "Bottleneck": kernels that split the key/value length across the GPU are
// the standard fix for this shape of work.  "33. Removing overhead", section "CUDA graphs for a changing
// batch": a row with length 0 (padding) must produce zeros, never NaN, and a graphed kernel must not
// take its grid from host-side batch values -- here the grid is (rows, kv_heads, max_splits) with
// max_splits fixed by the block-table width, and CTAs past a row's real length exit at once.
//
// Work of one CTA: request row, KV head, and a range of `split_blocks` 16-key blocks.  The G = Hq / Hkv
// query heads of the KV head share every K/V load: they are the rows of a 16-row MMA tile.  Each of the
// 4 warps takes every 4th block of the range (cp.async double buffering into an XOR-swizzled tile),
// computes S = Q K^T and O += P V with bf16 m16n8k16 MMAs and an online softmax in base 2.  Warps merge
// through shared memory; splits merge in the last-arriving CTA (atomic ticket, no waiting), always in
// split order, so the result does not depend on arrival order.
#include "common.cuh"
#include "kernels.h"

namespace grd {

template <int D>
__global__ void __launch_bounds__(128) k_attn_decode(AttnDecodeParams p) {
  constexpr int NCH = D / 8;  // 16-byte chunks per key row
  constexpr int KS = D / 16;  // k-steps of Q K^T
  constexpr int TILE = 16 * D;
  const int row = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.Hq / p.Hkv;
  const int h0 = kvh * G;

  const int r = p.r0 + row;
  const int sl = p.seq_lens[r];
  const int tok = p.cu[r];
  bf16* out = p.out + (size_t)tok * p.Hq * D + (size_t)h0 * D;
  int nblk = (sl + 15) >> 4;
  if (nblk > p.mbs) {  // never read past a block-table row
    if (split == 0 && threadIdx.x == 0) set_status(p.status, ST_BAD_POSITION);
    nblk = p.mbs;
  }
  const int nsplit = min((nblk + p.split_blocks - 1) / p.split_blocks, p.max_splits);
  if (sl <= 0) {  // padding row: zeros
    pdl_wait();
    if (split == 0)
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) out[i] = __float2bfloat16_rn(0.f);
    return;
  }
  if (split >= nsplit) return;
  const int b_begin = split * p.split_blocks;
  const int b_end = min(nblk, b_begin + p.split_blocks);

  extern __shared__ __align__(16) uint8_t smem[];
  bf16* wbuf = reinterpret_cast<bf16*>(smem) + warp * (4 * TILE);  // 2 stages x (K, V)

  float o[D / 8][4];
#pragma unroll
  for (int c = 0; c < D / 8; ++c) o[c][0] = o[c][1] = o[c][2] = o[c][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  auto issue = [&](int b, int stage) {
    int blk = p.bt[(size_t)r * p.mbs + b];
    if (blk < 0 || blk >= p.NB) {
      set_status(p.status, ST_BAD_BLOCK);
      blk = p.NB;
    }
    const bf16* ks_ = p.k_pool + ((size_t)blk * p.Hkv + kvh) * TILE;
    const bf16* vs_ = p.v_pool + ((size_t)blk * p.Hkv + kvh) * TILE;
    bf16* kd = wbuf + stage * 2 * TILE;
    bf16* vd = kd + TILE;
#pragma unroll
    for (int i = lane; i < 16 * NCH; i += 32) {
      const int rr = i / NCH, c = i % NCH;
      const int sw = (c ^ (rr & 7)) * 8;
      cp_async16(kd + rr * D + sw, ks_ + rr * D + c * 8);
      cp_async16(vd + rr * D + sw, vs_ + rr * D + c * 8);
    }
    cp_async_commit();
  };

  int b = b_begin + warp;
  int stage = 0;
  // context blocks already in the pool can be fetched before the preceding kernel finishes; the block that
  // holds this step's new token (the last one) is written by that kernel
  const bool early = b < b_end && b != nblk - 1;
  if (early) issue(b, 0);
  pdl_wait();
  if (b < b_end && !early) issue(b, 0);
  // Q fragments: rows = the G query heads (rows >= G are zero), k = head dimension
  uint32_t qa[KS][4];
  const bf16* qb = p.q + (size_t)tok * p.Hq * D + (size_t)h0 * D;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int d0 = ks * 16 + 2 * t;
    qa[ks][0] = (g < G) ? *reinterpret_cast<const uint32_t*>(qb + g * D + d0) : 0u;
    qa[ks][1] = (g + 8 < G) ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * D + d0) : 0u;
    qa[ks][2] = (g < G) ? *reinterpret_cast<const uint32_t*>(qb + g * D + d0 + 8) : 0u;
    qa[ks][3] = (g + 8 < G) ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * D + d0 + 8) : 0u;
  }

  for (; b < b_end; b += 4) {
    if (b + 4 < b_end) {
      issue(b + 4, stage ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const bf16* kt = wbuf + stage * 2 * TILE;
    const bf16* vt = kt + TILE;
    if (b == nblk - 1 && (sl & 15)) {
      // keys past the sequence get probability 0, but 0 * NaN is NaN: clear the stale V rows of the
      // last block (a reused block may hold anything there)
      const int first_bad = sl & 15;
      bf16* vw = wbuf + stage * 2 * TILE + TILE;
      for (int i = lane; i < (16 - first_bad) * NCH; i += 32) {
        const int rr = first_bad + i / NCH, c = i % NCH;
        *reinterpret_cast<uint4*>(vw + rr * D + ((c ^ (rr & 7)) * 8)) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }

    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        const int m = lane >> 3;
        const int kr = nt * 8 + (lane & 7);
        const int ch = 2 * (ks + (m >> 1)) + (m & 1);
        uint32_t bb[4];
        ldmatrix_x4(bb, kt + kr * D + ((ch ^ (kr & 7)) * 8));
        mma_bf16(sc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], bb[0], bb[1]);
        mma_bf16(sc[nt], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], bb[2], bb[3]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = b * 16 + nt * 8 + 2 * t + (j & 1);
        sc[nt][j] = (key < sl) ? sc[nt][j] * p.scale_log2 : -INFINITY;
      }
    float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = exp2f(sc[nt][0] - mn0);
      pr[nt][1] = exp2f(sc[nt][1] - mn0);
      pr[nt][2] = exp2f(sc[nt][2] - mn1);
      pr[nt][3] = exp2f(sc[nt][3] - mn1);
    }
    float s0 = pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
    float s1 = pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    l0 = l0 * a0 + s0;
    l1 = l1 * a1 + s1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      o[c][0] *= a0;
      o[c][1] *= a0;
      o[c][2] *= a1;
      o[c][3] *= a1;
    }
    const uint32_t pa0 = pack_bf16x2(pr[0][0], pr[0][1]);
    const uint32_t pa1 = pack_bf16x2(pr[0][2], pr[0][3]);
    const uint32_t pa2 = pack_bf16x2(pr[1][0], pr[1][1]);
    const uint32_t pa3 = pack_bf16x2(pr[1][2], pr[1][3]);
#pragma unroll
    for (int c = 0; c < D / 8; c += 2) {
      const int m = lane >> 3;
      const int vr = (m & 1) * 8 + (lane & 7);
      const int ch = c + (m >> 1);
      uint32_t bb[4];
      ldmatrix_x4_trans(bb, vt + vr * D + ((ch ^ (vr & 7)) * 8));
      mma_bf16(o[c], pa0, pa1, pa2, pa3, bb[0], bb[1]);
      mma_bf16(o[c + 1], pa0, pa1, pa2, pa3, bb[2], bb[3]);
    }
    __syncwarp();
    stage ^= 1;
  }

  // ---- merge the 4 warps (fixed order)
  __syncthreads();
  float* ms = reinterpret_cast<float*>(smem);  // [4][16]
  float* ls = ms + 64;                          // [4][16]
  float* os = ls + 64;                          // [4][16][D]
  if (t == 0) {
    ms[warp * 16 + g] = m0;
    ms[warp * 16 + g + 8] = m1;
    ls[warp * 16 + g] = l0;
    ls[warp * 16 + g + 8] = l1;
  }
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    float* r0 = os + (warp * 16 + g) * D + c * 8 + 2 * t;
    float* r8 = os + (warp * 16 + g + 8) * D + c * 8 + 2 * t;
    r0[0] = o[c][0];
    r0[1] = o[c][1];
    r8[0] = o[c][2];
    r8[1] = o[c][3];
  }
  __syncthreads();

  const bool single = nsplit == 1;
  float* part = p.ws + (((size_t)row * p.Hkv + kvh) * p.max_splits + split) * (size_t)G * (D + 2);
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int hr = i / D, dd = i - hr * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, ms[w * 16 + hr]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float sc_ = exp2f(ms[w * 16 + hr] - M);
      L += ls[w * 16 + hr] * sc_;
      O += os[(w * 16 + hr) * D + dd] * sc_;
    }
    if (single) {
      out[hr * D + dd] = __float2bfloat16_rn(O / L);
    } else {
      __stcg(part + hr * (D + 2) + dd, O);
      if (dd == 0) {
        __stcg(part + hr * (D + 2) + D, M);
        __stcg(part + hr * (D + 2) + D + 1, L);
      }
    }
  }
  if (single) return;

  // ---- split merge by the last CTA of (row, kv head), in split order
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* tk = p.tickets + (size_t)row * p.Hkv + kvh;
    const int old = atomicAdd(tk, 1);
    s_last = (old == nsplit - 1);
    if (s_last) *tk = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* base = p.ws + ((size_t)row * p.Hkv + kvh) * p.max_splits * (size_t)G * (D + 2);
  // split weights exp2(M_s - M) and the total L per head row, all loads in flight at once
  float* sw = reinterpret_cast<float*>(smem);   // [nsplit][G] weights
  float* sm = sw + p.max_splits * G;            // [G] merged max, then [G] 1 / L
  for (int i = threadIdx.x; i < nsplit * G; i += blockDim.x) {
    const int sp = i / G, hr = i - sp * G;
    sw[i] = __ldcg(base + ((size_t)sp * G + hr) * (D + 2) + D);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int hr = threadIdx.x;
    float M = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, sw[sp * G + hr]);
    float L = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
      const float w = exp2f(sw[sp * G + hr] - M);
      sw[sp * G + hr] = w;
      L += __ldcg(base + ((size_t)sp * G + hr) * (D + 2) + D + 1) * w;
    }
    sm[hr] = 1.f / L;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int hr = i / D, dd = i - hr * D;
    float O = 0.f;
#pragma unroll 8
    for (int sp = 0; sp < nsplit; ++sp) O += __ldcg(base + ((size_t)sp * G + hr) * (D + 2) + dd) * sw[sp * G + hr];
    out[hr * D + dd] = __float2bfloat16_rn(O * sm[hr]);
  }
}

size_t attn_decode_ws_floats(int rows, int Hq, int Hkv, int d, int max_splits) {
  const int G = Hq / Hkv;
  return (size_t)rows * Hkv * max_splits * G * (d + 2);
}

cudaError_t launch_attn_decode(const AttnDecodeParams& p, const LaunchOpts& o, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows, p.Hkv, p.max_splits);
  cfg.blockDim = dim3(128);
  const size_t tiles = (size_t)4 * 4 * 16 * p.d * 2;                  // 4 warps x 2 stages x (K, V)
  const size_t merge = (size_t)(128 + 4 * 16 * p.d) * 4;
  cfg.dynamicSmemBytes = tiles > merge ? tiles : merge;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.d == 128) {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(k_attn_decode<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
      set = true;
    }
    return cudaLaunchKernelEx(&cfg, k_attn_decode<128>, p);
  }
  if (p.d == 64) {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(k_attn_decode<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
      set = true;
    }
    return cudaLaunchKernelEx(&cfg, k_attn_decode<64>, p);
  }
  return cudaErrorInvalidValue;
}

}  // namespace grd
