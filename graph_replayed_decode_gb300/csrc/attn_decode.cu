// attn_decode.cu -- paged decode attention: one query row per request, split over the key length.
//
// "One forward per step", section "What changed": decode positions are reshaped to one query row per
// request so that every request's history is read in parallel (0.347 ms as rows vs 1.749 ms packed on
// the page's A10), and section "Bottleneck": kernels that split the key/value length across the GPU are
// the standard fix for this shape of work.  "33. Removing overhead", section "CUDA graphs for a changing
// batch": a row with length 0 (padding) must produce zeros, never NaN, and a graphed kernel must not
// take its grid from host-side batch values -- here the grid is (rows, kv_heads, splits) with the split
// count fixed by the block-table width, and CTAs past a row's real length do no work.
//
// Work of one CTA: request row, KV head, and a range of `split_blocks` 16-key blocks.  The G = Hq / Hkv
// (<= 8) query heads of the KV head share every K/V load: head g is row g of a 16-row MMA tile and row
// g + 8 carries the low half of its operand (q as bf16 hi/lo pairs in S = Q K^T, the probabilities as
// hi/lo pairs in O += P V, common.cuh), so both products keep fp32 operands at no extra MMA.  Each of the
// 4 warps takes every 4th block of the range (cp.async double buffering into an XOR-swizzled tile; blocks
// already in the pool are fetched before the kernel waits for the preceding kernel, only the block that
// holds this step's new token after), computes S = Q K^T and O += P V with bf16 m16n8k16 MMAs and an
// online softmax in base 2.  Warps merge through shared memory.  A split past the row's length (short
// rows in a batch sized for long ones) exits at once.  With several splits, each writes its unnormalised
// (O, max, sum) to a global workspace and counts itself in on an atomic counter; the split that finishes
// last merges all of them in split order and resets the counter, so the result does not depend on which
// split finishes last, and the next launch (or graph replay) finds the counter at zero.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace grd {

static constexpr int kStages = 2;    // K/V blocks in flight per warp
static constexpr int kMaxSplits = kAttnMaxSplits;  // splits of one (row, KV head)
static constexpr int kClusterSplits = 8;  // at most this many merge on chip (one thread-block cluster)

// Per-warp K/V stages, reused for the warp merge afterwards ([4][16] M, [4][16] L, [4][16][D] O, [G][D+2]).
__host__ __device__ constexpr size_t attn_stage_bytes(int D) {
  return (size_t)4 * kStages * 2 * 16 * D * 2 > (size_t)(128 + 4 * 16 * D + 16 * (D + 2)) * 4
             ? (size_t)4 * kStages * 2 * 16 * D * 2
             : (size_t)(128 + 4 * 16 * D + 16 * (D + 2)) * 4;
}

// Final merge of a row's split partials (O unnormalised, M, L per head), in split order, written as the
// output projection's operand planes.  get(sp, head, j) reads partial sp's value j (j < D: O, D: M,
// D + 1: L); the on-chip and the global-memory merges share this code, so they agree bit for bit.
template <int D, typename Get>
ENG_DEVICE void merge_splits(const AttnDecodeParams& p, int nsplit, int G, size_t obase, Get get) {
  // one output element per thread and iteration: its head's maxima and sums and its own partial sums of
  // every split are loaded together (one round trip when the partials sit in L2), then combined in split
  // order: M = max M_s, w_s = 2^(M_s - M), L = sum L_s w_s, out = (sum O_s w_s) / L
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int hr = i / D, dd = i - hr * D;
    float ms[kMaxSplits], ls[kMaxSplits], os[kMaxSplits];
#pragma unroll
    for (int sp = 0; sp < kMaxSplits; ++sp) {
      ms[sp] = sp < nsplit ? get(sp, hr, D) : -INFINITY;
      ls[sp] = sp < nsplit ? get(sp, hr, D + 1) : 0.f;
      os[sp] = sp < nsplit ? get(sp, hr, dd) : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < kMaxSplits; ++sp)
      if (sp < nsplit) M = fmaxf(M, ms[sp]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int sp = 0; sp < kMaxSplits; ++sp)
      if (sp < nsplit) {
        const float w = exp2f(ms[sp] - M);
        L += ls[sp] * w;
        O += os[sp] * w;
      }
    put_split(p.out_h, p.out_l, obase + hr * D + dd, O * (1.f / L));
  }
}

// Per-CTA scratch outside the dynamic K/V stages.
struct AttnShared {
  int last;
};

// One work item: split `split` of (row, KV head).  CLUSTER: the splits of a (row, KV head) are one
// thread-block cluster and split 0 merges them from its own shared memory (lowest latency; few rows).
// Otherwise partials go to the global workspace and the last split to finish merges them.
template <int D, bool CLUSTER>
ENG_DEVICE void attn_item(const AttnDecodeParams& p, int row, int kvh, int split, uint8_t* smem, AttnShared& sh) {
  constexpr int NCH = D / 8;  // 16-byte chunks per key row
  constexpr int KS = D / 16;  // k-steps of Q K^T
  constexpr int TILE = 16 * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.Hq / p.Hkv;
  const int h0 = kvh * G;
  int& s_last = sh.last;
  cg::cluster_group cluster = cg::this_cluster();

  // lengths and block tables are step inputs, final before the step's first kernel
  const int r = p.r0 + row;
  const int sl = p.seq_lens[r];
  const int tok = p.cu[r];
  const size_t obase = (size_t)tok * p.Hq * D + (size_t)h0 * D;  // this KV head's outputs (operand planes)
  int nblk = (sl + 15) >> 4;
  if (nblk > p.mbs) {  // never read past a block-table row
    if (split == 0 && threadIdx.x == 0) set_status(p.status, ST_BAD_POSITION);
    nblk = p.mbs;
  }
  const int nsplit = min((nblk + p.split_blocks - 1) / p.split_blocks, p.max_splits);
  const bool active = sl > 0 && split < nsplit;
  const int b_begin = split * p.split_blocks;
  const int b_end = min(nblk, b_begin + p.split_blocks);
  if (!CLUSTER && !active) {  // nothing to read: a padding row (zeros from split 0) or a split past its length
    pdl_trigger();
    if (sl <= 0 && split == 0) {
      pdl_wait();
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) put_split(p.out_h, p.out_l, obase + i, 0.f);
    }
    return;
  }

  bf16* wbuf = reinterpret_cast<bf16*>(smem) + warp * (kStages * 2 * TILE);  // kStages x (K, V) per warp

  float o[D / 8][4];
#pragma unroll
  for (int c = 0; c < D / 8; ++c) o[c][0] = o[c][1] = o[c][2] = o[c][3] = 0.f;
  float m0 = -INFINITY, l0 = 0.f;  // running max / sum of head g (rows g and g + 8 are its two halves)

  // this warp's blocks are b_begin + warp + 4 j; lane j holds the j-th one's pool id (block tables are
  // step inputs), so issuing a copy needs no dependent load
  const int nb = active && b_begin + warp < b_end ? (b_end - b_begin - warp + 3) / 4 : 0;
  int my_blk = 0;
  if (lane < nb) my_blk = p.bt[(size_t)r * p.mbs + b_begin + warp + 4 * lane];
  const uint64_t kv_pol = l2_evict_first();
  auto issue = [&](int b, int stage) {
    const int j = (b - b_begin - warp) >> 2;
    int blk = j < 32 ? __shfl_sync(0xffffffffu, my_blk, j & 31) : p.bt[(size_t)r * p.mbs + b];
    if (blk < 0 || blk >= p.NB) {
      set_status(p.status, ST_BAD_BLOCK);
      blk = p.NB;
    }
    const bf16* ks_ = p.k_pool + ((size_t)blk * p.Hkv + kvh) * TILE;
    const bf16* vs_ = p.v_pool + ((size_t)blk * p.Hkv + kvh) * TILE;
    bf16* kd = wbuf + (stage % kStages) * 2 * TILE;
    bf16* vd = kd + TILE;
#pragma unroll
    for (int i = lane; i < 16 * NCH; i += 32) {
      const int rr = i / NCH, c = i % NCH;
      const int sw = (c ^ (rr & 7)) * 8;
      cp_async16_hint(kd + rr * D + sw, ks_ + rr * D + c * 8, kv_pol);  // K/V are read once per step
      cp_async16_hint(vd + rr * D + sw, vs_ + rr * D + c * 8, kv_pol);
    }
    cp_async_commit();
  };

  // up to kStages of this warp's blocks in flight.  Blocks already in the pool are fetched before the
  // kernel waits for the preceding kernel; the block that holds this step's new token (the sequence's
  // last block) only after.
  const int ahead = min(nb, kStages);
  int issued = 0;
  for (; issued < ahead; ++issued) {
    const int bb = b_begin + warp + 4 * issued;
    if (bb == nblk - 1) break;
    issue(bb, issued);
  }
  if (CLUSTER && p.max_splits > 1) cluster.sync();  // every split has started before pushes into split 0
  pdl_trigger();
  pdl_wait();
  for (; issued < ahead; ++issued) issue(b_begin + warp + 4 * issued, issued);

  uint32_t qa[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) qa[ks][0] = qa[ks][1] = qa[ks][2] = qa[ks][3] = 0u;
  if (active && g < G) {  // Q fragments: row g = hi of head g, row g + 8 = its lo (rows of heads >= G: zero)
    const float* qb = p.q + (size_t)tok * p.Hq * D + (size_t)(h0 + g) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = ks * 16 + 2 * t;
      const float2 x0 = *reinterpret_cast<const float2*>(qb + d0);
      const float2 x1 = *reinterpret_cast<const float2*>(qb + d0 + 8);
      split_bf16x2(x0.x, x0.y, qa[ks][0], qa[ks][1]);
      split_bf16x2(x1.x, x1.y, qa[ks][2], qa[ks][3]);
    }
  }

  for (int j = 0; j < nb; ++j) {
    const int b = b_begin + warp + 4 * j;
    const int stage = j % kStages;
    switch (issued - j - 1) {  // block j has landed once at most this many later groups are pending
      case 0: cp_async_wait<0>(); break;
      case 1: cp_async_wait<1>(); break;
      default: cp_async_wait<2>(); break;
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
    // head g's score of key nt * 8 + 2 t + j: its hi row (j) plus its lo row (j + 2)
    float sv[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = b * 16 + nt * 8 + 2 * t + j;
        sv[nt][j] = (key < sl) ? (sc[nt][j] + sc[nt][j + 2]) * p.scale_log2 : -INFINITY;
      }
    float mx = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m0, mx);  // finite: the block holds at least one key < sl
    const float a0 = exp2f(m0 - mn);
    float pr[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = exp2f(sv[nt][0] - mn);
      pr[nt][1] = exp2f(sv[nt][1] - mn);
    }
    float s0 = pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    l0 = l0 * a0 + s0;
    m0 = mn;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      o[c][0] *= a0;
      o[c][1] *= a0;
      o[c][2] *= a0;
      o[c][3] *= a0;
    }
    // P fragments: row g = hi of the probabilities, row g + 8 = lo
    uint32_t pa0, pa1, pa2, pa3;
    split_bf16x2(pr[0][0], pr[0][1], pa0, pa1);
    split_bf16x2(pr[1][0], pr[1][1], pa2, pa3);
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
    if (issued < nb) {  // refill the stage just consumed
      issue(b_begin + warp + 4 * issued, issued % kStages);
      ++issued;
    }
  }

  // ---- merge the 4 warps (fixed order) into this CTA's partial [G][D + 2] = (O, M, L)
  __syncthreads();
  float* ms = reinterpret_cast<float*>(smem);  // [4][16]
  float* ls = ms + 64;                          // [4][16]
  float* os = ls + 64;                          // [4][16][D]
  if (t == 0) {
    ms[warp * 16 + g] = m0;
    ls[warp * 16 + g] = l0;
  }
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {  // head g's output: hi row + lo row
    float* r0 = os + (warp * 16 + g) * D + c * 8 + 2 * t;
    r0[0] = o[c][0] + o[c][2];
    r0[1] = o[c][1] + o[c][3];
  }
  __syncthreads();
  // this CTA's partial (O unnormalised, M, L) of head hr, element dd
  auto partial = [&](int hr, int dd, float& O, float& M, float& L) {
    M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, ms[w * 16 + hr]);
    L = 0.f;
    O = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float sc_ = exp2f(ms[w * 16 + hr] - M);
      L += ls[w * 16 + hr] * sc_;
      O += os[(w * 16 + hr) * D + dd] * sc_;
    }
  };

  if (CLUSTER) {
    float* recv = reinterpret_cast<float*>(smem + attn_stage_bytes(D));  // split 0: [splits][G][D + 2]
    if (active) {
      float* dst = nsplit > 1 ? cluster.map_shared_rank(recv, 0) + (size_t)split * G * (D + 2) : nullptr;
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int hr = i / D, dd = i - hr * D;
        float O, M, L;
        partial(hr, dd, O, M, L);
        if (nsplit == 1) {
          put_split(p.out_h, p.out_l, obase + hr * D + dd, O / L);
        } else {  // push this split's partial into split 0's receive buffer
          dst[hr * (D + 2) + dd] = O;
          if (dd == 0) {
            dst[hr * (D + 2) + D] = M;
            dst[hr * (D + 2) + D + 1] = L;
          }
        }
      }
    } else if (sl <= 0 && split == 0) {  // padding row: zeros
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) put_split(p.out_h, p.out_l, obase + i, 0.f);
    }
    if (p.max_splits > 1) {
      cluster.sync();
      if (split == 0 && sl > 0 && nsplit > 1)
        merge_splits<D>(p, nsplit, G, obase,
                        [&](int sp, int hr, int j) { return recv[((size_t)sp * G + hr) * (D + 2) + j]; });
    }
    return;
  }

  float* part = p.ws + (((size_t)row * p.Hkv + kvh) * p.max_splits + split) * G * (D + 2);
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int hr = i / D, dd = i - hr * D;
    float O, M, L;
    partial(hr, dd, O, M, L);
    if (nsplit == 1) {
      put_split(p.out_h, p.out_l, obase + hr * D + dd, O / L);
    } else {  // this split's unnormalised partial (O, M, L)
      part[hr * (D + 2) + dd] = O;
      if (dd == 0) {
        part[hr * (D + 2) + D] = M;
        part[hr * (D + 2) + D + 1] = L;
      }
    }
  }
  if (nsplit == 1) return;

  // ---- the last split to finish merges the partials in split order
  __threadfence();
  __syncthreads();
  int* counter = p.counters + (size_t)row * p.Hkv + kvh;
  if (threadIdx.x == 0) s_last = atomicAdd(counter, 1) == nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* parts = p.ws + ((size_t)row * p.Hkv + kvh) * p.max_splits * G * (D + 2);
  merge_splits<D>(p, nsplit, G, obase,
                  [&](int sp, int hr, int j) { return __ldcg(parts + ((size_t)sp * G + hr) * (D + 2) + j); });
  if (threadIdx.x == 0) *counter = 0;  // ready for the next launch
}

// Few rows: one CTA per (row, KV head, split), the splits of a (row, KV head) in one cluster.
template <int D>
__global__ void __launch_bounds__(128) k_attn_decode_cluster(AttnDecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ AttnShared sh;
  if (threadIdx.x == 0 && p.pf_bytes) prefetch_share(p.pf_ptr, p.pf_bytes);
  attn_item<D, true>(p, blockIdx.x, blockIdx.y, blockIdx.z, smem, sh);
}

// Many rows: one CTA per (row, KV head, split) slot of the capture-frozen grid; slots past a row's length
// exit at once, and partials merge through the global workspace.
template <int D>
__global__ void __launch_bounds__(128) k_attn_decode_global(AttnDecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ AttnShared sh;
  if (threadIdx.x == 0 && p.pf_bytes) prefetch_share(p.pf_ptr, p.pf_bytes);
  attn_item<D, false>(p, blockIdx.x, blockIdx.y, blockIdx.z, smem, sh);
}

template <typename K>
static cudaError_t launch_kernel(K kernel, cudaLaunchConfig_t& cfg, const AttnDecodeParams& p) {
  const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kernel), 200 * 1024);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_attn_decode(const AttnDecodeParams& p, const LaunchOpts& o, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  if (p.max_splits < 1 || p.max_splits > kMaxSplits || p.Hq / p.Hkv > 8) return cudaErrorInvalidValue;
  if (p.d != 64 && p.d != 128) return cudaErrorInvalidValue;
  // a few rows: merge on chip (a cluster per row and KV head); many rows: the global workspace, so that
  // splits past a short row's length leave their SM at once
  const bool cluster = p.rows <= 4 && p.max_splits <= kClusterSplits;
  if (!cluster && p.max_splits > 1 && (!p.ws || !p.counters)) return cudaErrorInvalidValue;
  const int G = p.Hq / p.Hkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows, p.Hkv, p.max_splits);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = attn_stage_bytes(p.d) + (cluster ? (size_t)kClusterSplits * G * (p.d + 2) * 4 : 0);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = p.max_splits;
  cfg.attrs = attr;
  cfg.numAttrs = cluster && p.max_splits > 1 ? 2 : 1;
  if (cluster)
    return p.d == 128 ? launch_kernel(k_attn_decode_cluster<128>, cfg, p)
                      : launch_kernel(k_attn_decode_cluster<64>, cfg, p);
  return p.d == 128 ? launch_kernel(k_attn_decode_global<128>, cfg, p)
                    : launch_kernel(k_attn_decode_global<64>, cfg, p);
}

}  // namespace grd
