// moe.cu -- a mixture-of-experts MLP whose shapes never depend on the routing.
//
// "33. Removing overhead", section "A MoE layer that never asks the host": instead of one matmul per
// expert and a host-side count of each expert's tokens, the assignments (token, slot) are grouped by expert
// on the device, each group padded to whole blocks of BLOCK_M rows, and a grouped GEMM multiplies every
// block by the weights of the expert that owns it.  Every launch's grid depends only on the token count N,
// the experts per token k, the expert count E and BLOCK_M, so the whole layer can sit in a CUDA graph.
//
//   k_moe_route    router logits x W_r^T (fp32 accumulation of the bf16 operands), softmax, the k most
//                  probable experts with ties to the lower id, their probabilities renormalised to sum to 1
//                  (the reading of Qwen3-MoE's router; the pages call it from a chapter not included);
//   k_moe_align    counts per expert, padded group offsets, the assignments of each group in ascending
//                  order, each block's expert and the rows the groups occupy;
//   k_moe_gate_up  per block of 16 assignment rows and 32 activation columns: the token rows times the
//                  expert's gate and up rows (bf16 tensor-core MMAs, fp32 accumulation), silu(gate) * up
//                  written as bf16 hi/lo planes of the assignment rows;
//   k_moe_down     per block and 64 output columns: the activation planes times the expert's down rows
//                  (hi and lo products), scaled by the assignment's router weight;
//   k_moe_combine  each token's k assignment rows summed in slot order.
// Blocks past the rows the groups occupy (read from device memory) exit at once, and padding rows are
// neither read nor written, so a graph replay needs no host value of the routing.
#include "common.cuh"
#include "kernels.h"

namespace grd {

namespace {

constexpr int kMoeBm = 16;       // rows of a block (one MMA row tile)
constexpr int kMoeKb = 64;       // k-block of the grouped GEMMs' pipeline
constexpr int kMoeStages = 3;    // k-blocks in flight (cp.async)
constexpr int kMoeStride = kMoeKb + 8;  // padded row stride of a staged tile (bf16), 144 bytes
constexpr int kMoeStagedIds = 8192;     // the alignment keeps at most this many ids in shared memory
constexpr int kMoeMaxExperts = 1024;

ENG_DEVICE void ldsm_x4(uint32_t r[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// ------------------------------------------------------------------ router

// One CTA of 128 threads per token: logit e = x . W_r[e] (warp w takes experts w, w + 4, ...; lanes stride
// over the hidden size in 16-byte pieces and the warp sums in a fixed tree), then warp 0 takes the softmax
// and the top k.
__global__ void __launch_bounds__(128) k_moe_route(const bf16* __restrict__ x, const bf16* __restrict__ wr, int D,
                                                   int E, int k, float* __restrict__ w_out, int* __restrict__ id_out) {
  extern __shared__ float s_logit[];  // [E]
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * D);
  for (int e = warp; e < E; e += 4) {
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * D);
    float acc = 0.f;
    for (int i = lane; i < D / 8; i += 32) {
      const uint4 a = xr[i], b = wrow[i];
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 fa = unpack_bf16x2(av[j]), fb = unpack_bf16x2(bv[j]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) s_logit[e] = acc;
  }
  __syncthreads();
  if (warp != 0) return;
  float mx = -INFINITY;
  for (int e = lane; e < E; e += 32) mx = fmaxf(mx, s_logit[e]);
  mx = warp_max(mx);
  float sum = 0.f;
  for (int e = lane; e < E; e += 32) {
    const float pe = expf(s_logit[e] - mx);
    s_logit[e] = pe;
    sum += pe;
  }
  sum = warp_sum(sum);
  __syncwarp();
  // k rounds of a warp argmax over the probabilities not taken yet (ties to the lower id)
  float chosen = 0.f, wsel = 0.f;
  int isel = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -1.f;
    int bi = E;
    for (int e = lane; e < E; e += 32) {
      const float v = s_logit[e];
      if (v > bv) {  // ascending e: the first maximum of this lane is its lowest id
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi >= E) bi = 0, bv = 0.f;  // only with non-finite logits (every comparison false)
    if (lane == j) {
      wsel = bv / sum;
      isel = bi;
    }
    chosen += bv / sum;
    __syncwarp();
    if (lane == 0) s_logit[bi] = -2.f;  // taken
    __syncwarp();
  }
  if (lane < k) {
    w_out[(size_t)t * k + lane] = wsel / chosen;
    id_out[(size_t)t * k + lane] = isel;
  }
}

// ------------------------------------------------------------------ alignment

// One CTA of 1024 threads.  M = padded_rows(N k, E, bm) rows: sorted_ids[i] is the assignment a = token k +
// slot that row i handles (N k on a padding row); groups in expert order, ascending inside a group;
// block_expert[b] = the expert owning block b (E - 1 past the groups); out[0] = rows the groups occupy,
// out[1] = assignments whose expert id is out of range (placed nowhere).
__global__ void __launch_bounds__(1024) k_moe_align(const int* __restrict__ gids, int total, int E, int bm, int M,
                                                    bool staged, int* __restrict__ sorted_ids,
                                                    int* __restrict__ block_expert, int* __restrict__ out) {
  extern __shared__ int s_cnt[];  // [E] counts, [E + 1] padded offsets, then the ids when staged
  int* s_off = s_cnt + E;
  int* s_ids = s_off + E + 1;
  __shared__ int s_bad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
  if (tid == 0) s_bad = 0;
  for (int i = tid; i < M; i += blockDim.x) sorted_ids[i] = total;
  if (staged)
    for (int a = tid; a < total; a += blockDim.x) s_ids[a] = gids[a];
  const int* ids = staged ? s_ids : gids;
  __syncthreads();
  for (int a = tid; a < total; a += blockDim.x) {
    const int e = ids[a];
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    else atomicAdd(&s_bad, 1);
  }
  __syncthreads();
  if (tid == 0) {  // padded group offsets (E is small)
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_off[e] = acc;
      acc += (s_cnt[e] + bm - 1) / bm * bm;
    }
    s_off[E] = acc;
  }
  __syncthreads();
  // each warp places its experts' assignments in ascending order: one ballot per 32 assignments
  for (int e = warp; e < E; e += blockDim.x / 32) {
    int pos = s_off[e];
    for (int base = 0; base < total; base += 32) {
      const int a = base + lane;
      const bool mine = a < total && ids[a] == e;
      const unsigned m = __ballot_sync(0xffffffffu, mine);
      if (mine) sorted_ids[pos + __popc(m & ((1u << lane) - 1u))] = a;
      pos += __popc(m);
    }
  }
  for (int b = tid; b < M / bm; b += blockDim.x) {
    int e = E - 1;
    const int row = b * bm;
    if (row < s_off[E]) {  // the last group starting at or before this row
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= row) lo = mid;
        else hi = mid - 1;
      }
      e = lo;
    }
    block_expert[b] = e;
  }
  if (tid == 0) {
    out[0] = s_off[E];
    out[1] = s_bad;
  }
}

// ------------------------------------------------------------------ grouped GEMMs

// Shared tiles of one pipeline stage: the block's 16 rows and the 64 weight rows of the CTA, each 64 k.
struct MoeStage {
  bf16 a[kMoeBm * kMoeStride];
  bf16 a2[kMoeBm * kMoeStride];  // the lo plane (down projection only)
  bf16 w[64 * kMoeStride];
};

// Block b, activation columns [32 c, 32 c + 32): rows = the block's assignments, weight rows = the expert's
// gate rows 32 c .. 32 c + 31 (tile rows 0..31) and up rows I + 32 c .. (tile rows 32..63).  Warp w takes
// gate rows 8 w .. 8 w + 7 and the matching up rows, so silu(gate) * up stays in its registers.
__global__ void __launch_bounds__(128) k_moe_gate_up(const bf16* __restrict__ x, const bf16* __restrict__ gate_up,
                                                     const int* __restrict__ sorted_ids,
                                                     const int* __restrict__ block_expert,
                                                     const int* __restrict__ padded, int k, int total, int D, int I,
                                                     bf16* __restrict__ act_h, bf16* __restrict__ act_l) {
  extern __shared__ __align__(16) uint8_t smem[];
  MoeStage* st = reinterpret_cast<MoeStage*>(smem);
  __shared__ int s_row[kMoeBm];  // assignment of each row (total: padding)
  const int b = blockIdx.x, c = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (b * kMoeBm >= *padded) return;  // past the groups
  const int e = block_expert[b];
  if (tid < kMoeBm) s_row[tid] = sorted_ids[b * kMoeBm + tid];
  __syncthreads();
  const bf16* W = gate_up + (size_t)e * 2 * I * D;
  const int nkb = D / kMoeKb;
  auto issue = [&](int kb, int s) {
    MoeStage& S = st[s];
    {  // 16 rows x 8 pieces of 16 bytes: one piece a thread
      const int r = tid >> 3, pc = tid & 7;
      const int a = s_row[r];
      if (a < total) cp_async16(S.a + r * kMoeStride + pc * 8, x + (size_t)(a / k) * D + kb * kMoeKb + pc * 8);
    }
#pragma unroll
    for (int i = tid; i < 64 * 8; i += 128) {  // 64 weight rows x 8 pieces
      const int r = i >> 3, pc = i & 7;
      const int wrow = r < 32 ? 32 * c + r : I + 32 * c + (r - 32);
      cp_async16(S.w + r * kMoeStride + pc * 8, W + (size_t)wrow * D + kb * kMoeKb + pc * 8);
    }
    cp_async_commit();
  };
  for (int s = 0; s < kMoeStages - 1; ++s)
    if (s < nkb) issue(s, s);
    else cp_async_commit();
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // gate tile, up tile
  for (int kb = 0; kb < nkb; ++kb) {
    cp_async_wait<kMoeStages - 2>();
    __syncthreads();
    if (kb + kMoeStages - 1 < nkb) issue(kb + kMoeStages - 1, (kb + kMoeStages - 1) % kMoeStages);
    else cp_async_commit();
    const MoeStage& S = st[kb % kMoeStages];
#pragma unroll
    for (int ks = 0; ks < kMoeKb / 16; ++ks) {
      uint32_t af[4], bf[4];
      ldsm_x4(af, S.a + (lane & 15) * kMoeStride + ks * 16 + (lane >> 4) * 8);
      // lanes 0-15: gate rows 8 w + (lane & 7) at k 0 / 8; lanes 16-31: the matching up rows
      const int wr = (lane < 16 ? 8 * warp : 32 + 8 * warp) + (lane & 7);
      ldsm_x4(bf, S.w + wr * kMoeStride + ks * 16 + ((lane >> 3) & 1) * 8);
      mma_bf16(acc[0], af[0], af[1], af[2], af[3], bf[0], bf[1]);
      mma_bf16(acc[1], af[0], af[1], af[2], af[3], bf[2], bf[3]);
    }
  }
  cp_async_wait<0>();
  // fragment (row g, col 2 t), (g, 2 t + 1), (g + 8, 2 t), (g + 8, 2 t + 1): rows are assignments, cols are
  // activation columns 32 c + 8 w + col
  const int g = lane >> 2, t2 = 2 * (lane & 3);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int a = s_row[g + 8 * h];
    if (a >= total) continue;
    const size_t o = (size_t)a * I + 32 * c + 8 * warp + t2;
    const float g0 = acc[0][2 * h], g1 = acc[0][2 * h + 1], u0 = acc[1][2 * h], u1 = acc[1][2 * h + 1];
    put_split2(act_h, act_l, o, g0 / (1.f + expf(-g0)) * u0, g1 / (1.f + expf(-g1)) * u1);
  }
}

// Block b, output columns [64 c, 64 c + 64): the activation planes of the block's assignments times the
// expert's down rows (hi and lo products), scaled by each assignment's router weight.  Warp w takes output
// columns 64 c + 16 w .. + 15 (two MMA column tiles).
__global__ void __launch_bounds__(128) k_moe_down(const bf16* __restrict__ act_h, const bf16* __restrict__ act_l,
                                                  const bf16* __restrict__ down, const float* __restrict__ rw,
                                                  const int* __restrict__ sorted_ids,
                                                  const int* __restrict__ block_expert, const int* __restrict__ padded,
                                                  int total, int D, int I, float* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t smem[];
  MoeStage* st = reinterpret_cast<MoeStage*>(smem);
  __shared__ int s_row[kMoeBm];
  const int b = blockIdx.x, c = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (b * kMoeBm >= *padded) return;
  const int e = block_expert[b];
  if (tid < kMoeBm) s_row[tid] = sorted_ids[b * kMoeBm + tid];
  __syncthreads();
  const bf16* W = down + (size_t)e * D * I;
  const int nkb = I / kMoeKb;
  auto issue = [&](int kb, int s) {
    MoeStage& S = st[s];
    {
      const int r = tid >> 3, pc = tid & 7;
      const int a = s_row[r];
      if (a < total) {
        cp_async16(S.a + r * kMoeStride + pc * 8, act_h + (size_t)a * I + kb * kMoeKb + pc * 8);
        cp_async16(S.a2 + r * kMoeStride + pc * 8, act_l + (size_t)a * I + kb * kMoeKb + pc * 8);
      }
    }
#pragma unroll
    for (int i = tid; i < 64 * 8; i += 128) {
      const int r = i >> 3, pc = i & 7;
      cp_async16(S.w + r * kMoeStride + pc * 8, W + (size_t)(64 * c + r) * I + kb * kMoeKb + pc * 8);
    }
    cp_async_commit();
  };
  for (int s = 0; s < kMoeStages - 1; ++s)
    if (s < nkb) issue(s, s);
    else cp_async_commit();
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  float acl[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // lo-plane products, added at the end
  for (int kb = 0; kb < nkb; ++kb) {
    cp_async_wait<kMoeStages - 2>();
    __syncthreads();
    if (kb + kMoeStages - 1 < nkb) issue(kb + kMoeStages - 1, (kb + kMoeStages - 1) % kMoeStages);
    else cp_async_commit();
    const MoeStage& S = st[kb % kMoeStages];
#pragma unroll
    for (int ks = 0; ks < kMoeKb / 16; ++ks) {
      uint32_t ah[4], al[4], bf[4];
      ldsm_x4(ah, S.a + (lane & 15) * kMoeStride + ks * 16 + (lane >> 4) * 8);
      ldsm_x4(al, S.a2 + (lane & 15) * kMoeStride + ks * 16 + (lane >> 4) * 8);
      // lanes 0-15: output rows 16 w + (lane & 7) (tile 0), lanes 16-31: rows 16 w + 8 + (lane & 7) (tile 1)
      ldsm_x4(bf, S.w + (16 * warp + (lane >> 4) * 8 + (lane & 7)) * kMoeStride + ks * 16 + ((lane >> 3) & 1) * 8);
      mma_bf16(acc[0], ah[0], ah[1], ah[2], ah[3], bf[0], bf[1]);
      mma_bf16(acc[1], ah[0], ah[1], ah[2], ah[3], bf[2], bf[3]);
      mma_bf16(acl[0], al[0], al[1], al[2], al[3], bf[0], bf[1]);
      mma_bf16(acl[1], al[0], al[1], al[2], al[3], bf[2], bf[3]);
    }
  }
  cp_async_wait<0>();
  const int g = lane >> 2, t2 = 2 * (lane & 3);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int a = s_row[g + 8 * h];
    if (a >= total) continue;
    const float wgt = rw[a];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const size_t o = (size_t)a * D + 64 * c + 16 * warp + 8 * j + t2;
      y[o] = (acc[j][2 * h] + acl[j][2 * h]) * wgt;
      y[o + 1] = (acc[j][2 * h + 1] + acl[j][2 * h + 1]) * wgt;
    }
  }
}

// out[t] = sum over slots j (in order) of y[t k + j]
__global__ void k_moe_combine(const float* __restrict__ y, int N, int k, int D, float* __restrict__ out) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)N * D) return;
  const size_t t = i / D, d = i - t * D;
  float s = 0.f;
  for (int j = 0; j < k; ++j) s += y[(t * k + j) * D + d];
  out[i] = s;
}

}  // namespace

int moe_padded_rows(int total, int E, int bm) {
  const long long m = (long long)total + (long long)E * (bm - 1);
  return (int)((m + bm - 1) / bm * bm);
}

cudaError_t launch_moe_route(const bf16* x, const bf16* wr, int N, int D, int E, int k, float* w, int* ids,
                             cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  if (D % 8 || E < 1 || E > 4096 || k < 1 || k > 32 || k > E) return cudaErrorInvalidValue;
  k_moe_route<<<N, 128, (size_t)E * 4, s>>>(x, wr, D, E, k, w, ids);
  return cudaGetLastError();
}

cudaError_t launch_moe_align(const int* ids, int total, int E, int bm, int* sorted_ids, int* block_expert, int* out,
                             cudaStream_t s) {
  if (total < 0 || E < 1 || E > kMoeMaxExperts || bm < 1) return cudaErrorInvalidValue;
  const int M = moe_padded_rows(total, E, bm);
  const bool staged = total <= kMoeStagedIds;  // the ids in shared memory: every warp scans them per expert
  static_assert(kMoeStagedIds * 4 + (2 * kMoeMaxExperts + 1) * 4 <= 48 * 1024, "align kernel shared memory");
  k_moe_align<<<1, 1024, (size_t)(2 * E + 1 + (staged ? total : 0)) * 4, s>>>(ids, total, E, bm, M, staged, sorted_ids,
                                                                              block_expert, out);
  return cudaGetLastError();
}

size_t moe_workspace_bytes(int N, int k, int E, int D, int I) {
  const size_t total = (size_t)N * k, M = (size_t)moe_padded_rows((int)total, E, kMoeBm);
  return (M + M / kMoeBm + 4) * 4 + total * I * 2 * 2 + total * D * 4 + 256 * 4;
}

cudaError_t launch_moe_mlp(const bf16* x, const bf16* gate_up, const bf16* down, const float* rw, const int* ids,
                           int N, int D, int I, int E, int k, float* out, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  if (D % 64 || I % 64 || E < 1 || E > kMoeMaxExperts || k < 1 || !ws || ws_bytes < moe_workspace_bytes(N, k, E, D, I))
    return cudaErrorInvalidValue;
  const int total = N * k, M = moe_padded_rows(total, E, kMoeBm);
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  uint8_t* p = static_cast<uint8_t*>(ws);
  int* sorted_ids = reinterpret_cast<int*>(p);
  p += up((size_t)M * 4);
  int* block_expert = reinterpret_cast<int*>(p);
  p += up((size_t)(M / kMoeBm) * 4);
  int* info = reinterpret_cast<int*>(p);
  p += 256;
  bf16* act_h = reinterpret_cast<bf16*>(p);
  p += up((size_t)total * I * 2);
  bf16* act_l = reinterpret_cast<bf16*>(p);
  p += up((size_t)total * I * 2);
  float* y = reinterpret_cast<float*>(p);
  if (static_cast<size_t>(p - static_cast<uint8_t*>(ws)) + (size_t)total * D * 4 > ws_bytes)
    return cudaErrorInvalidValue;
  cudaError_t r = launch_moe_align(ids, total, E, kMoeBm, sorted_ids, block_expert, info, s);
  if (r != cudaSuccess) return r;
  // an assignment whose expert id is out of range is placed in no group: its rows stay zero
  if ((r = cudaMemsetAsync(y, 0, (size_t)total * D * 4, s)) != cudaSuccess) return r;
  const size_t smem = (size_t)kMoeStages * sizeof(MoeStage);
  k_moe_gate_up<<<dim3(M / kMoeBm, I / 32), 128, smem, s>>>(x, gate_up, sorted_ids, block_expert, info, k, total, D, I,
                                                            act_h, act_l);
  if ((r = cudaGetLastError()) != cudaSuccess) return r;
  k_moe_down<<<dim3(M / kMoeBm, D / 64), 128, smem, s>>>(act_h, act_l, down, rw, sorted_ids, block_expert, info, total,
                                                         D, I, y);
  if ((r = cudaGetLastError()) != cudaSuccess) return r;
  const size_t nd = (size_t)N * D;
  k_moe_combine<<<(unsigned)((nd + 255) / 256), 256, 0, s>>>(y, N, k, D, out);
  return cudaGetLastError();
}

}  // namespace grd
