// attn_decode.cu -- paged decode attention: one query row per request, split over the key length.
//
// "One forward per step", section "What changed": decode positions are reshaped to one query row per
// request so that every request's history is read in parallel (0.347 ms as rows vs 1.749 ms packed on
// the page's A10), and section "Bottleneck": kernels that split the key/value length across the GPU are
// the standard fix for this shape of work.  "33. Removing overhead", section "CUDA graphs for a changing
// batch": a row with length 0 (padding) must produce zeros, never NaN, and a graphed kernel must not
// take its grid from host-side batch values -- here every grid is fixed by the bucket and the engine
// (rows x KV heads x a split count fixed by the block-table width, or the flat partition's resident
// CTAs), and work past a row's real length is skipped.
//
// The G = Hq / Hkv (<= 8) query heads of a KV head share every K/V load: head g is row g of a 16-row
// MMA tile and row g + 8 carries the low half of its operand (q as 16-bit hi/lo pairs in S = Q K^T, the
// probabilities as hi/lo pairs in O += P V, common.cuh), so both products keep fp32 operands at no extra
// MMA.  A warp streams 16-key blocks through two cp.async stages (XOR-swizzled rows), computes S and
// O += P V with m16n8k16 MMAs of the element type and keeps an online softmax in base 2.  Blocks already
// in the pool are fetched before the kernel waits for the preceding kernel, only the block that holds
// this step's new token after.  Three launch shapes:
//   * a few rows (<= 4): a CTA per (row, KV head, split), the splits of a row in one thread-block
//     cluster, merged on chip in split order;
//   * more rows, a KV head serving at most two query heads: a fixed grid of CTAs over a flat partition of
//     all the rows' blocks (k_attn_decode_flat below), so that rows of very different lengths still keep
//     every SM streaming to the end;
//   * more rows, larger query groups: a CTA per (row, KV head, split), merged through a global workspace.
// All merge partial results in a fixed order, so the result does not depend on which CTA or warp finishes
// last, and every counter is back at zero when the launch ends (graph replay finds it so).
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace grd {
ENG_ELEM_NS_BEGIN

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

// ---- per-block pieces shared by both kernels (one warp, one 16-key block of one (row, KV head))

// The K and V rows of one pool block into a warp's stage (row rr's 16-byte chunk c at chunk c ^ (rr & 7),
// so that the fragment loads below are free of bank conflicts); one commit group.  K/V are read once per
// step, so the copies carry an evict-first L2 policy.
template <int D>
ENG_DEVICE void attn_copy_block(bf16* kd, const bf16* ks, const bf16* vs, int lane, uint64_t pol) {
  constexpr int NCH = D / 8;
  bf16* vd = kd + 16 * D;
#pragma unroll
  for (int i = lane; i < 16 * NCH; i += 32) {
    const int rr = i / NCH, c = i % NCH;
    const int sw = (c ^ (rr & 7)) * 8;
    cp_async16_hint(kd + rr * D + sw, ks + rr * D + c * 8, pol);
    cp_async16_hint(vd + rr * D + sw, vs + rr * D + c * 8, pol);
  }
  cp_async_commit();
}

// Keys past the sequence get probability 0, but 0 * NaN is NaN: the stale V rows of a sequence's last
// block (a reused block may hold anything there) are cleared before use.
template <int D>
ENG_DEVICE void attn_clear_tail(bf16* vt, int sl, int lane) {
  constexpr int NCH = D / 8;
  const int first_bad = sl & 15;
  for (int i = lane; i < (16 - first_bad) * NCH; i += 32) {
    const int rr = first_bad + i / NCH, c = i % NCH;
    *reinterpret_cast<uint4*>(vt + rr * D + ((c ^ (rr & 7)) * 8)) = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncwarp();
}

// Q fragments of the G query heads of one KV head: row g = hi of head g, row g + 8 = its lo (rows of
// heads >= G: zero).  qb points at head 0 of the group.
template <int D>
ENG_DEVICE void attn_load_q(const float* qb, int G, int lane, uint32_t (&qa)[D / 16][4]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) qa[ks][0] = qa[ks][1] = qa[ks][2] = qa[ks][3] = 0u;
  if (g < G) {
    const float* q = qb + (size_t)g * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int d0 = ks * 16 + 2 * t;
      const float2 x0 = *reinterpret_cast<const float2*>(q + d0);
      const float2 x1 = *reinterpret_cast<const float2*>(q + d0 + 8);
      split_bf16x2(x0.x, x0.y, qa[ks][0], qa[ks][1]);
      split_bf16x2(x1.x, x1.y, qa[ks][2], qa[ks][3]);
    }
  }
}

// One block (keys key0 .. key0 + 15 of a sequence of sl keys): S = Q K^T, the online softmax update of
// (m0, l0) in base 2, and O = alpha O + P V.  The probabilities enter P V as hi/lo rows like q.
template <int D>
ENG_DEVICE void attn_block(const bf16* kt, const bf16* vt, int key0, int sl, float scale_log2,
                           const uint32_t (&qa)[D / 16][4], float (&o)[D / 8][4], float& m0, float& l0, int lane) {
  constexpr int KS = D / 16;
  const int t = lane & 3;
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
      const int key = key0 + nt * 8 + 2 * t + j;
      sv[nt][j] = (key < sl) ? (sc[nt][j] + sc[nt][j + 2]) * scale_log2 : -INFINITY;
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
}

// Pool address of block b of request r (a bad id is reported and replaced by the scratch block).
ENG_DEVICE int attn_pool_block(const AttnDecodeParams& p, int r, int b) {
  int blk = p.bt[(size_t)r * p.mbs + b];
  if (blk < 0 || blk >= p.NB) {
    set_status(p.status, ST_BAD_BLOCK);
    blk = p.NB;
  }
  return blk;
}

// ---- one CTA per (row, KV head, split)

// Work of one CTA: request row, KV head, and a range of `split_blocks` 16-key blocks.  Each of the 4
// warps takes every 4th block of the range (cp.async double buffering; blocks already in the pool are
// fetched before the kernel waits for the preceding kernel, only the block that holds this step's new
// token after).  Warps merge through shared memory.  CLUSTER: the splits of a row form a thread-block
// cluster and merge on split 0 through distributed shared memory (a few rows).  Otherwise each split
// writes its unnormalised (O, max, sum) to a global workspace and counts itself in on an atomic counter;
// the split that finishes last merges them, in split order, and resets the counter (rows whose KV heads
// serve more than two query heads, where the flat partition's merges cost more than they save).
template <int D, bool CLUSTER>
__global__ void __launch_bounds__(128) k_attn_decode_split(AttnDecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_last;
  constexpr int TILE = 16 * D;
  const int row = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.Hq / p.Hkv;
  const int h0 = kvh * G;
  cg::cluster_group cluster = cg::this_cluster();
  if (threadIdx.x == 0 && p.pf_bytes) prefetch_share(p.pf_ptr, p.pf_bytes);

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
    attn_copy_block<D>(wbuf + (stage % kStages) * 2 * TILE, p.k_pool + ((size_t)blk * p.Hkv + kvh) * TILE,
                       p.v_pool + ((size_t)blk * p.Hkv + kvh) * TILE, lane, kv_pol);
  };

  // up to kStages of this warp's blocks in flight
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

  uint32_t qa[D / 16][4];
  attn_load_q<D>(p.q + (size_t)tok * p.Hq * D + (size_t)h0 * D, active ? G : 0, lane, qa);

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
    if (b == nblk - 1 && (sl & 15)) attn_clear_tail<D>(wbuf + stage * 2 * TILE + TILE, sl, lane);
    attn_block<D>(kt, vt, b * 16, sl, p.scale_log2, qa, o, m0, l0, lane);
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

  if (!CLUSTER) {
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
    // the last split to finish merges the partials in split order
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
    return;
  }
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
}

// ---- many rows: the flat partition
//
// The K/V blocks of every (row, KV head) segment of the launch are laid end to end -- row by row, KV
// head by KV head, each segment preceded by kSegUnits units that stand for its fixed cost (the query
// load and the partial write) -- and every warp of the grid takes an equal contiguous range of the
// units, so every warp streams about the same number of bytes whatever the mix of lengths (a grid of
// (row, KV head, split) CTAs leaves the long rows' last splits running alone at the end of the launch).
// A warp streams its range through its two stages, carrying the online softmax across the blocks of one
// segment.  Where a segment ends inside its range, or its range ends inside a segment, it closes a piece:
// a segment that one warp covers is written out directly; otherwise every piece writes (O, M, L) and
// the piece that finishes last merges the segment's pieces in piece order.  The partition depends only
// on the step's lengths and the grid size, so a launch on the same inputs always adds the same terms in
// the same order.
static constexpr int kSegUnits = 2;  // about a piece's fixed cost, in blocks
static constexpr int kMergeBatch = 16;  // pieces whose loads are in flight together in a merge

// Shared arrays of the flat kernel after the warps' stages: per row its block count (0 for a padding
// row), length and query token, then the first unit of each row and the total.
__host__ __device__ constexpr size_t flat_smem_bytes(int D, int rows) {
  return attn_stage_bytes(D) + (size_t)(4 * rows + 1) * 4;
}

template <int D>
__global__ void __launch_bounds__(128) k_attn_decode_flat(AttnDecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int TILE = 16 * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.Hq / p.Hkv, Hkv = p.Hkv, R = p.rows;
  int* s_nblk = reinterpret_cast<int*>(smem + attn_stage_bytes(D));
  int* s_sl = s_nblk + R;
  int* s_tok = s_sl + R;
  int* s_base = s_tok + R;  // [R + 1]
  if (threadIdx.x == 0 && p.pf_bytes) prefetch_share(p.pf_ptr, p.pf_bytes);

  // rows (step inputs, final before the step's first kernel)
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int sl = p.seq_lens[p.r0 + r];
    int nb = sl > 0 ? (sl + 15) >> 4 : 0;
    if (nb > p.mbs) {  // never read past a block-table row
      if (blockIdx.x == 0) set_status(p.status, ST_BAD_POSITION);
      nb = p.mbs;
    }
    s_nblk[r] = nb;
    s_sl[r] = sl;
    s_tok[r] = p.cu[p.r0 + r];
  }
  __syncthreads();
  if (warp == 0) {  // first unit of each row: exclusive prefix of Hkv (kSegUnits + blocks), 32 rows at a time
    int run = 0;
    for (int c0 = 0; c0 < R; c0 += 32) {
      const int r = c0 + lane;
      const int u = (r < R && s_nblk[r] > 0) ? Hkv * (kSegUnits + s_nblk[r]) : 0;
      int x = u;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (r < R) s_base[r] = run + x - u;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_base[R] = run;
  }
  __syncthreads();
  pdl_trigger();

  const int W = s_base[R];
  const int NWe = min((int)gridDim.x * 4, W);  // warps with work: ranges of at least one unit
  const int gw = blockIdx.x * 4 + warp;
  if (gw >= NWe) {
    pdl_wait();
  } else {
    const int A = (int)((long long)gw * W / NWe), B = (int)((long long)(gw + 1) * W / NWe);
    // the segment of unit A: the last row whose first unit is <= A (rows of no blocks have no units)
    int lo = 0, hi = R;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_base[mid] <= A) lo = mid;
      else hi = mid;
    }
    auto unit_of = [&](int r, int h, int b) {
      return r < R ? s_base[r] + h * (kSegUnits + s_nblk[r]) + kSegUnits + b : W;
    };
    auto advance = [&](int& r, int& h, int& b) {
      if (++b == s_nblk[r]) {
        b = 0;
        if (++h == Hkv) {
          h = 0;
          do ++r; while (r < R && s_nblk[r] == 0);
        }
      }
    };
    int cr = lo, ch, cb;  // compute cursor: (row, KV head, block) of the next block to compute
    {
      const int seg = kSegUnits + s_nblk[cr], off = A - s_base[cr];
      ch = off / seg;
      cb = max(0, off - ch * seg - kSegUnits);
    }
    int ir = cr, ih = ch, ib = cb;  // issue cursor
    bf16* wbuf = reinterpret_cast<bf16*>(smem) + warp * (kStages * 2 * TILE);
    const uint64_t kv_pol = l2_evict_first();
    // pool ids of this warp's blocks, 32 at a time: lane j holds the id of block (batch * 32 + j)
    int my_blk = 0, batch_first = 0;
    auto load_batch = [&](int r, int h, int b) {
      for (int j = 0; j < lane; ++j) {
        if (r >= R) break;
        advance(r, h, b);
      }
      my_blk = (r < R && unit_of(r, h, b) < B) ? attn_pool_block(p, p.r0 + r, b) : p.NB;
    };
    int issued = 0;
    auto issue = [&]() {
      if ((issued & 31) == 0 && issued > batch_first) {
        load_batch(ir, ih, ib);
        batch_first = issued;
      }
      const int blk = __shfl_sync(0xffffffffu, my_blk, issued & 31);
      attn_copy_block<D>(wbuf + (issued % kStages) * 2 * TILE, p.k_pool + ((size_t)blk * Hkv + ih) * TILE,
                         p.v_pool + ((size_t)blk * Hkv + ih) * TILE, lane, kv_pol);
      advance(ir, ih, ib);
      ++issued;
    };
    load_batch(ir, ih, ib);
    // blocks already in the pool are fetched before the kernel waits for the preceding kernel; the block
    // that holds this step's new token (a segment's last block) only after
    while (issued < kStages && unit_of(ir, ih, ib) < B && ib != s_nblk[ir] - 1) issue();
    pdl_wait();
    while (issued < kStages && unit_of(ir, ih, ib) < B) issue();

    uint32_t qa[D / 16][4];
    float o[D / 8][4];
    float m0 = -INFINITY, l0 = 0.f;
    for (int j = 0; unit_of(cr, ch, cb) < B; ++j) {
      if (j == 0 || cb == 0) {  // a piece starts: its query rows, a fresh softmax
        attn_load_q<D>(p.q + ((size_t)s_tok[cr] * p.Hq + (size_t)ch * G) * D, G, lane, qa);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) o[c][0] = o[c][1] = o[c][2] = o[c][3] = 0.f;
        m0 = -INFINITY;
        l0 = 0.f;
      }
      switch (issued - j - 1) {  // block j has landed once at most this many later groups are pending
        case 0: cp_async_wait<0>(); break;
        default: cp_async_wait<1>(); break;
      }
      __syncwarp();
      const int sl = s_sl[cr], nblk = s_nblk[cr];
      bf16* kt = wbuf + (j % kStages) * 2 * TILE;
      if (cb == nblk - 1 && (sl & 15)) attn_clear_tail<D>(kt + TILE, sl, lane);
      attn_block<D>(kt, kt + TILE, cb * 16, sl, p.scale_log2, qa, o, m0, l0, lane);
      __syncwarp();
      if (unit_of(ir, ih, ib) < B) issue();  // refill the stage just consumed

      const int r = cr, h = ch;
      advance(cr, ch, cb);
      if (cb != 0 && unit_of(cr, ch, cb) < B) continue;  // the piece goes on
      // ---- close the piece of segment (r, h)
      const int s = r * Hkv + h;
      const int S0 = unit_of(r, h, 0), S1 = S0 + nblk;
      const int wf = (int)(((long long)(S0 + 1) * NWe - 1) / W), wl = (int)(((long long)S1 * NWe - 1) / W);
      const int np = wl - wf + 1;
      const size_t obase = ((size_t)s_tok[r] * p.Hq + (size_t)h * G) * D;
      if (np == 1) {  // the whole segment: normalised output
        if (g < G) {
          const float inv = 1.f / l0;
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
#pragma unroll
            for (int k = 0; k < 2; ++k)
              put_split(p.out_h, p.out_l, obase + (size_t)g * D + c * 8 + 2 * t + k, (o[c][k] + o[c][k + 2]) * inv);
        }
        continue;
      }
      // piece gw - wf of the segment: slot s + wf + piece (distinct over all segments of the launch)
      float* part = p.ws + (size_t)(s + gw) * G * (D + 2);
      if (g < G) {
        float* pg = part + (size_t)g * (D + 2);
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
#pragma unroll
          for (int k = 0; k < 2; ++k) pg[c * 8 + 2 * t + k] = o[c][k] + o[c][k + 2];
        if (t == 0) {
          pg[D] = m0;
          pg[D + 1] = l0;
        }
      }
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(p.counters + s, 1) == np - 1;
      if (!__shfl_sync(0xffffffffu, last, 0)) continue;
      __threadfence();
      // the last piece merges them all, in piece order: M = max M_q, w_q = 2^(M_q - M),
      // out = (sum_q O_q w_q) / (sum_q L_q w_q), each head's outputs kMergeBatch pieces at a time (a few
      // round trips to L2 for a segment of dozens of pieces); lane j holds elements 2 j, 2 j + 1 (+ 64 i)
      const size_t PS = (size_t)G * (D + 2);  // floats per piece
      for (int hr = 0; hr < G; ++hr) {
        const float* bh = p.ws + (size_t)(s + wf) * PS + (size_t)hr * (D + 2);
        float mx = -INFINITY, lq = 0.f, mq_l = -INFINITY;
        for (int q = lane; q < np; q += 32) mx = fmaxf(mx, __ldcg(bh + q * PS + D));
        mx = warp_max(mx);
        for (int q = lane; q < np; q += 32) {
          mq_l = __ldcg(bh + q * PS + D);
          lq += __ldcg(bh + q * PS + D + 1) * exp2f(mq_l - mx);
        }
        const float inv = 1.f / warp_sum(lq);
        float2 acc[D / 64];
#pragma unroll
        for (int i = 0; i < D / 64; ++i) acc[i] = make_float2(0.f, 0.f);
        for (int q0 = 0; q0 < np; q0 += kMergeBatch) {
          float mq[kMergeBatch];
          float2 v[kMergeBatch][D / 64];
#pragma unroll
          for (int k = 0; k < kMergeBatch; ++k) {
            const bool in = q0 + k < np;
            const float* pq = bh + (size_t)(q0 + k) * PS;
            mq[k] = in ? __ldcg(pq + D) : -INFINITY;
#pragma unroll
            for (int i = 0; i < D / 64; ++i)
              v[k][i] = in ? __ldcg(reinterpret_cast<const float2*>(pq + 64 * i + 2 * lane)) : make_float2(0.f, 0.f);
          }
#pragma unroll
          for (int k = 0; k < kMergeBatch; ++k) {
            const float w = q0 + k < np ? exp2f(mq[k] - mx) : 0.f;
#pragma unroll
            for (int i = 0; i < D / 64; ++i) {
              acc[i].x += v[k][i].x * w;
              acc[i].y += v[k][i].y * w;
            }
          }
        }
        const size_t ob = obase + (size_t)hr * D;
#pragma unroll
        for (int i = 0; i < D / 64; ++i) put_split2(p.out_h, p.out_l, ob + 64 * i + 2 * lane, acc[i].x * inv, acc[i].y * inv);
      }
      if (lane == 0) p.counters[s] = 0;  // ready for the next launch
    }
  }
  // padding rows (no keys): zeros, a CTA per row
  for (int r = blockIdx.x; r < R; r += gridDim.x)
    if (s_nblk[r] == 0)
      for (int i = threadIdx.x; i < p.Hq * D; i += blockDim.x)
        put_split(p.out_h, p.out_l, (size_t)s_tok[r] * p.Hq * D + i, 0.f);
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
  // a few rows: merge on chip (a cluster per row and KV head); more rows: the flat partition when a KV head
  // serves at most two query heads, else splits merged through the workspace.  Only the row count and the
  // shape decide, and 4 is a default capture size, so an eager step and its padded bucket take the same
  // kernel.
  const int G = p.Hq / p.Hkv;
  const bool cluster = p.rows <= 4 && p.max_splits <= kClusterSplits;
  const bool flat = !cluster && G <= 2;
  if (!cluster && (!p.ws || !p.counters || (flat && p.flat_ctas < 1))) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (flat) {
    cfg.gridDim = dim3(p.flat_ctas);
    cfg.dynamicSmemBytes = flat_smem_bytes(p.d, p.rows);
    return p.d == 128 ? launch_kernel(k_attn_decode_flat<128>, cfg, p) : launch_kernel(k_attn_decode_flat<64>, cfg, p);
  }
  cfg.gridDim = dim3(p.rows, p.Hkv, p.max_splits);
  if (!cluster) {
    cfg.dynamicSmemBytes = attn_stage_bytes(p.d);
    return p.d == 128 ? launch_kernel(k_attn_decode_split<128, false>, cfg, p)
                      : launch_kernel(k_attn_decode_split<64, false>, cfg, p);
  }
  cfg.dynamicSmemBytes = attn_stage_bytes(p.d) + (size_t)kClusterSplits * G * (p.d + 2) * 4;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = p.max_splits;
  cfg.numAttrs = p.max_splits > 1 ? 2 : 1;
  return p.d == 128 ? launch_kernel(k_attn_decode_split<128, true>, cfg, p)
                    : launch_kernel(k_attn_decode_split<64, true>, cfg, p);
}

int attn_flat_ctas(int d, int rows, int sms) {
  const void* k = d == 128 ? reinterpret_cast<const void*>(k_attn_decode_flat<128>)
                           : reinterpret_cast<const void*>(k_attn_decode_flat<64>);
  const size_t smem = flat_smem_bytes(d, rows);
  if (ensure_smem_limit(k, 200 * 1024) != cudaSuccess) return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 128, smem) != cudaSuccess) return 0;
  // two CTAs (8 warps, 16 blocks in flight) per SM keep HBM busy; more warps only cut the segments into
  // more pieces to merge (batch-32 decode of the 0.6B shape: 2.36 ms/step at two, 2.40 at three)
  return (per_sm < 2 ? per_sm : 2) * sms;
}

ENG_ELEM_NS_END
}  // namespace grd
