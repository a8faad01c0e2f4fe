// attn_prefill.cu -- packed causal attention for the prefill chunks of a step.
//
// "One forward per step", section "What changed": chunk positions stay packed and run a causal prefill
// kernel over the paged cache; the chunk's own K/V were written to the pool by the preceding KV-write
// kernel, earlier chunks of the same prompt are already there.  A query at position p sees keys 0..p of
// its own request ("19. Fast decode", section "Static shapes and a static cache": key_pos <= query_pos).
//
// One CTA per (work item, query head): a work item is up to 64 consecutive query tokens of one request;
// its 4 warps own 16 query rows each.  Keys stream through shared memory 64 at a time (4 paged blocks,
// cp.async double buffering, XOR-swizzled 16-byte chunks); S = Q K^T and O += P V use bf16 m16n8k16 MMAs
// with an online softmax in base 2.  Q and P enter the products as bf16 hi/lo pairs (common.cuh): one MMA
// per half, so both keep fp32 operands.  Key rows past the chunk's last position are zero-filled so that
// masked (zero) probabilities never meet stale NaN values.
#include "common.cuh"
#include "kernels.h"

namespace grd {
ENG_ELEM_NS_BEGIN

template <int D>
__global__ void __launch_bounds__(128) k_attn_prefill(AttnPrefillParams p) {
  constexpr int NCH = D / 8;
  constexpr int KS = D / 16;
  constexpr int KT = 64;  // keys per tile
  constexpr int TILE = KT * D;
  const int item = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.Hq / p.Hkv, kvh = h / G;

  pdl_wait();
  const int4 it = p.items[item];
  const int r = it.x, first = it.y, count = it.z;
  const int maxpos = p.positions[first + count - 1];
  const int nkeys = maxpos + 1;
  const int ntiles = (nkeys + KT - 1) / KT;

  const int rb = 16 * warp;
  const bool v0 = rb + g < count, v8 = rb + g + 8 < count;
  const int qp0 = v0 ? p.positions[first + rb + g] : maxpos;
  const int qp8 = v8 ? p.positions[first + rb + g + 8] : maxpos;
  const int warp_max = (rb < count) ? p.positions[first + min(count - 1, rb + 15)] : -1;

  uint32_t qa[KS][4], ql[KS][4];  // hi and lo fragments of the warp's 16 query rows
  const float* q0 = p.q + ((size_t)(first + rb + g) * p.Hq + h) * D;
  const float* q8 = p.q + ((size_t)(first + rb + g + 8) * p.Hq + h) * D;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int d0 = ks * 16 + 2 * t;
    const float2 z = make_float2(0.f, 0.f);
    const float2 a0 = v0 ? *reinterpret_cast<const float2*>(q0 + d0) : z;
    const float2 a8 = v8 ? *reinterpret_cast<const float2*>(q8 + d0) : z;
    const float2 b0 = v0 ? *reinterpret_cast<const float2*>(q0 + d0 + 8) : z;
    const float2 b8 = v8 ? *reinterpret_cast<const float2*>(q8 + d0 + 8) : z;
    split_bf16x2(a0.x, a0.y, qa[ks][0], ql[ks][0]);
    split_bf16x2(a8.x, a8.y, qa[ks][1], ql[ks][1]);
    split_bf16x2(b0.x, b0.y, qa[ks][2], ql[ks][2]);
    split_bf16x2(b8.x, b8.y, qa[ks][3], ql[ks][3]);
  }

  extern __shared__ __align__(16) uint8_t smem[];
  bf16* buf = reinterpret_cast<bf16*>(smem);  // [2 stages][K tile, V tile]

  auto issue = [&](int tile, int stage) {
    bf16* kd = buf + stage * 2 * TILE;
    bf16* vd = kd + TILE;
    for (int i = threadIdx.x; i < KT * NCH; i += blockDim.x) {
      const int rr = i / NCH, c = i % NCH;
      const int key = tile * KT + rr;
      const int sw = (c ^ (rr & 7)) * 8;
      if (key < nkeys) {
        int blk = p.bt[(size_t)r * p.mbs + (key >> 4)];
        if (blk < 0 || blk >= p.NB) {
          set_status(p.status, ST_BAD_BLOCK);
          blk = p.NB;
        }
        const size_t src = (((size_t)blk * p.Hkv + kvh) * 16 + (key & 15)) * D + c * 8;
        cp_async16(kd + rr * D + sw, p.k_pool + src);
        cp_async16(vd + rr * D + sw, p.v_pool + src);
      } else {
        *reinterpret_cast<uint4*>(kd + rr * D + sw) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(vd + rr * D + sw) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_async_commit();
  };

  float o[D / 8][4];
#pragma unroll
  for (int c = 0; c < D / 8; ++c) o[c][0] = o[c][1] = o[c][2] = o[c][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  issue(0, 0);
  for (int tile = 0; tile < ntiles; ++tile) {
    const int stage = tile & 1;
    if (tile + 1 < ntiles) {
      issue(tile + 1, stage ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const bf16* kt = buf + stage * 2 * TILE;
    const bf16* vt = kt + TILE;
    if (tile * KT <= warp_max) {
      float sc[8][4], sl[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        sl[nt][0] = sl[nt][1] = sl[nt][2] = sl[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ks += 2) {
          const int m = lane >> 3;
          const int kr = nt * 8 + (lane & 7);
          const int ch = 2 * (ks + (m >> 1)) + (m & 1);
          uint32_t bb[4];
          ldmatrix_x4(bb, kt + kr * D + ((ch ^ (kr & 7)) * 8));
          mma_bf16(sc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], bb[0], bb[1]);
          mma_bf16(sl[nt], ql[ks][0], ql[ks][1], ql[ks][2], ql[ks][3], bb[0], bb[1]);
          mma_bf16(sc[nt], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], bb[2], bb[3]);
          mma_bf16(sl[nt], ql[ks + 1][0], ql[ks + 1][1], ql[ks + 1][2], ql[ks + 1][3], bb[2], bb[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[nt][j] += sl[nt][j];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int key = tile * KT + nt * 8 + 2 * t;
        sc[nt][0] = (key <= qp0) ? sc[nt][0] * p.scale_log2 : -INFINITY;
        sc[nt][1] = (key + 1 <= qp0) ? sc[nt][1] * p.scale_log2 : -INFINITY;
        sc[nt][2] = (key <= qp8) ? sc[nt][2] * p.scale_log2 : -INFINITY;
        sc[nt][3] = (key + 1 <= qp8) ? sc[nt][3] * p.scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      // a row whose keys in this tile are all masked keeps its state (mn = m, scale 1)
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float a0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
      const float a1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = (mn0 == -INFINITY) ? 0.f : exp2f(sc[nt][0] - mn0);
        sc[nt][1] = (mn0 == -INFINITY) ? 0.f : exp2f(sc[nt][1] - mn0);
        sc[nt][2] = (mn1 == -INFINITY) ? 0.f : exp2f(sc[nt][2] - mn1);
        sc[nt][3] = (mn1 == -INFINITY) ? 0.f : exp2f(sc[nt][3] - mn1);
        s0 += sc[nt][0] + sc[nt][1];
        s1 += sc[nt][2] + sc[nt][3];
      }
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
#pragma unroll
      for (int kk = 0; kk < KT / 16; ++kk) {
        uint32_t pa0, pa1, pa2, pa3, pl0, pl1, pl2, pl3;
        split_bf16x2(sc[2 * kk][0], sc[2 * kk][1], pa0, pl0);
        split_bf16x2(sc[2 * kk][2], sc[2 * kk][3], pa1, pl1);
        split_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1], pa2, pl2);
        split_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3], pa3, pl3);
#pragma unroll
        for (int c = 0; c < D / 8; c += 2) {
          const int m = lane >> 3;
          const int vr = kk * 16 + (m & 1) * 8 + (lane & 7);
          const int ch = c + (m >> 1);
          uint32_t bb[4];
          ldmatrix_x4_trans(bb, vt + vr * D + ((ch ^ (vr & 7)) * 8));
          mma_bf16(o[c], pa0, pa1, pa2, pa3, bb[0], bb[1]);
          mma_bf16(o[c], pl0, pl1, pl2, pl3, bb[0], bb[1]);
          mma_bf16(o[c + 1], pa0, pa1, pa2, pa3, bb[2], bb[3]);
          mma_bf16(o[c + 1], pl0, pl1, pl2, pl3, bb[2], bb[3]);
        }
      }
    }
    __syncthreads();
  }

  // rows: g (o[c][0..1]) and g + 8 (o[c][2..3]); l is already summed over the 4 lanes of a row
  const float i0 = (l0 > 0.f) ? 1.f / l0 : 0.f;
  const float i8 = (l1 > 0.f) ? 1.f / l1 : 0.f;
  const size_t out0 = ((size_t)(first + rb + g) * p.Hq + h) * D;  // rows g and g + 8 in the operand planes
  const size_t out8 = ((size_t)(first + rb + g + 8) * p.Hq + h) * D;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const int d = c * 8 + 2 * t;
    if (v0) put_split2(p.out_h, p.out_l, out0 + d, o[c][0] * i0, o[c][1] * i0);
    if (v8) put_split2(p.out_h, p.out_l, out8 + d, o[c][2] * i8, o[c][3] * i8);
  }
}

cudaError_t launch_attn_prefill(const AttnPrefillParams& p, const LaunchOpts& o, cudaStream_t s) {
  if (p.n_items <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_items, p.Hq);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = (size_t)2 * 2 * 64 * p.d * 2;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.d == 128) {
    const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(k_attn_prefill<128>), 96 * 1024);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, k_attn_prefill<128>, p);
  }
  if (p.d == 64) return cudaLaunchKernelEx(&cfg, k_attn_prefill<64>, p);
  return cudaErrorInvalidValue;
}

ENG_ELEM_NS_END
}  // namespace grd
