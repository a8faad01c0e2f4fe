// gemm.cu -- skinny GEMM Y[T][N] = X[T][K] . W[N][K]^T for the decode-sized projections, with the
// step's norms and elementwise work fused into its prologue and epilogue.
//
// Shapes: T is the packed token count of the step (1..64 in decode, larger in prefill, handled in
// 64-token chunks), N the output width, K the reduction width.  "33. Removing overhead", section "Fewer,
// larger matmuls": Q/K/V and gate/up are each one matmul over a concatenated matrix; add_norm does the
// residual add and the next norm in one memory pass; and the fusions production engines use -- SiLU-and-mul,
// RoPE inside the KV write, the LM head with sampling -- save a pass over memory and a launch each.
//
// At decode sizes the kernel is bound by the latency of its dependent memory round trips, not by
// bandwidth, so the design minimises the work left after the previous kernel finishes:
//   * W is pre-packed in m16n8k16 fragment order (common.cuh).  Before waiting for its inputs
//     (griddepcontrol.wait) every warp loads its first k-tiles' A fragments into registers and the CTA
//     asks L2 to prefetch the rest of its slice, so weight streaming overlaps the preceding kernel;
//   * X arrives as two bf16 planes hi = bf16(x) and lo = bf16(x - hi) (common.cuh), written by the
//     producing kernel; every weight fragment meets both, into two fp32 accumulators added at the end, so
//     the product keeps fp32 activations to about 2^-16.  After the wait, warp 0 bulk-copies each token's
//     rows of the CTA's K-range into shared memory (one copy per row and plane, in one piece when it fits)
//     and the warps read them with ldmatrix;
//   * a norm before the GEMM costs no pass: the producer of the residual h writes the planes of h * w
//     (w the norm weight) and per-row-group partial sums of h^2, and since RMSNorm(h) W^T equals
//     (1 / rms(h)) ((h * w) W^T), the kernel scales each token's outputs by its 1 / rms, computed from the
//     partial sums while the copies are in flight;
//   * a CTA owns RG 16-row tiles and one of S K-ranges; its 8 warps split the K-range and sum in a fixed
//     order; the S CTAs of a row group form a thread-block cluster and add their tiles through distributed
//     shared memory, always in split order (each CTA finishing a block of consecutive tokens) --
//     deterministic and independent of T, so graph replay and eager execution are bit-identical;
//   * epilogues run over the finished [16 RG rows x tokens] tile in shared memory:
//       EPI_STORE_F32  out = Y (+bias)
//       EPI_RESID      h += Y, each token's sum of h^2 over this CTA's rows and the planes of h * w_next
//                      (for the next norm and GEMM)
//       EPI_SILU       planes of silu(gate) * up, on row-interleaved gate|up tiles
//       EPI_QKV_ROPE   the CTA's rows are whole heads: +bias, per-head QK-RMSNorm, rotate-half RoPE, and the
//                      paged KV write (q heads -> q buffer, k/v heads -> pool slot of the token)
//       EPI_LMHEAD     logits (optional) and a per-token (key, index) maximum for greedy / Gumbel-max
//                      sampling; the last CTA turns the maxima into token ids.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace cg = cooperative_groups;

namespace grd {
ENG_ELEM_NS_BEGIN

static constexpr int kPieceTiles = 16;          // k-tiles (x32 columns) per X piece when X does not fit whole
static constexpr int kPreMax = 8;               // k-tiles per warp loaded into registers before waiting
static constexpr size_t kWholeXBytes = 128 * 1024;  // both planes
static constexpr int kMaxClusterDev = 8;        // largest split-K cluster
static constexpr int kCsTokens = 8;             // tokens whose RoPE row is staged before the wait

// Shared-memory plan of one launch (host and device agree on it).  When the CTA's weight slice is at most
// kTmaMaxBytes it is bulk-copied (TMA) into shared memory before the kernel waits for its inputs; the X
// staging area and the reduction tiles follow it.
struct GemmSmem {
  int piece;       // k-tiles of X staged per piece
  bool tma;        // weights staged in shared memory
  size_t w_bytes;  // weight slice (0 unless tma)
  size_t x_bytes;  // X staging: hi plane, then lo plane, [NT * 8 rows][piece * 32 + 8] each
  size_t red_bytes;
  size_t ts_bytes;
  size_t recv_bytes;
  size_t recv_off;  // offset of the receive buffer inside the staging area
  size_t total;
};

static constexpr size_t kTmaMaxBytes = 128 * 1024;
static constexpr size_t kSmemBudget = 200 * 1024;     // dynamic shared memory a tensor-core GEMM CTA may use
static constexpr size_t kSmemBudgetMma = 216 * 1024;  // and a warp-MMA one (its static arrays take under 8 KB)

// Split-K: CTA `split` of a cluster finishes the block of kblk consecutive tokens starting at split * kblk
// (a multiple of 4, so that partial sums move between CTAs as 16-byte vectors).
__host__ __device__ inline int gemm_kblk(int NT, int S) {
  const int k = (NT * 8 + S - 1) / S;
  return (k + 3) & ~3;
}

__host__ __device__ inline GemmSmem gemm_smem(int NT, int RG, int ktn, int S) {
  GemmSmem m;
  const size_t whole = (size_t)2 * NT * 8 * (ktn * 32 + 8) * 2;
  m.piece = whole <= kWholeXBytes ? ktn : (ktn < kPieceTiles ? ktn : kPieceTiles);
  const size_t w = (size_t)RG * ktn * 1024;
  m.tma = w <= kTmaMaxBytes;
  m.w_bytes = m.tma ? w : 0;
  m.x_bytes = (size_t)2 * NT * 8 * (m.piece * 32 + 8) * 2;
  m.red_bytes = (size_t)8 * NT * 32 * 16;
  m.ts_bytes = (size_t)16 * RG * (NT * 8 + 1) * 4;
  // split-K: every CTA pushes its tile's columns for the tokens another CTA finishes into that CTA's
  // receive buffer [S][16 RG rows][tokens per CTA]
  m.recv_bytes = S > 1 ? (size_t)S * 16 * RG * gemm_kblk(NT, S) * 4 : 0;
  const size_t tail = m.red_bytes + m.ts_bytes;
  // the receive buffer gets its own space: peers push into it while this CTA may still be staging X or
  // reducing its own tile
  m.recv_off = m.x_bytes > tail ? m.x_bytes : tail;
  m.recv_off = (m.recv_off + 15) & ~(size_t)15;
  m.total = m.w_bytes + m.recv_off + m.recv_bytes;
  if (m.tma && m.total > kSmemBudgetMma) {  // too big with the weights staged: stream them through registers
    m.tma = false;
    m.total -= m.w_bytes;
    m.w_bytes = 0;
  }
  return m;
}

template <int NT>
ENG_DEVICE void mma_tile(float (&acc)[NT][4], float (&accl)[NT][4], const uint4& a0, const uint4& a1, const bf16* xs,
                         const bf16* xl, int xstride, int kt, int lane) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    uint32_t b[4], bl[4];
    const int m = lane >> 3;
    const int off = (nt * 8 + (lane & 7)) * xstride + kt * 32 + (m >> 1) * 16 + (m & 1) * 8;
    ldmatrix_x4(b, xs + off);
    ldmatrix_x4(bl, xl + off);
    mma_bf16(acc[nt], a0.x, a0.y, a0.z, a0.w, b[0], b[1]);
    mma_bf16(accl[nt], a0.x, a0.y, a0.z, a0.w, bl[0], bl[1]);
    mma_bf16(acc[nt], a1.x, a1.y, a1.z, a1.w, b[2], b[3]);
    mma_bf16(accl[nt], a1.x, a1.y, a1.z, a1.w, bl[2], bl[3]);
  }
}

ENG_DEVICE float4 scale4(const float4 a, float rs, const float4 w) {
  return make_float4(a.x * rs * w.x, a.y * rs * w.y, a.z * rs * w.z, a.w * rs * w.w);
}

// Eight consecutive fp32 activations -> the hi and lo planes at element index idx.
ENG_DEVICE void stage8(bf16* xs, bf16* xl, int idx, const float4 a, const float4 b) {
  uint4 h, l;
  split_bf16x2(a.x, a.y, h.x, l.x);
  split_bf16x2(a.z, a.w, h.y, l.y);
  split_bf16x2(b.x, b.y, h.z, l.z);
  split_bf16x2(b.z, b.w, h.w, l.w);
  *reinterpret_cast<uint4*>(xs + idx) = h;
  *reinterpret_cast<uint4*>(xl + idx) = l;
}

// Tensor-core path (TC): 64-token chunks against 128-row weight tiles, k-blocks of 64 through a ring of
// kTcStages shared-memory stages (weight tile, hi tile, lo tile per stage, TMA tensor copies with 128-byte
// swizzle); one thread issues two tcgen05 MMAs per 16 k (hi plane, lo plane) into a 128 x 64 fp32 TMEM
// accumulator; the accumulator is read back into the same [rows][tokens] tile the epilogues use.
static constexpr int kTcStages = 3;
static constexpr uint32_t kTcA = 128 * 128;           // 128 weight rows x 64 bf16
static constexpr uint32_t kTcB = 64 * 128;            // 64 tokens x 64 bf16, one plane
static constexpr uint32_t kTcStage = kTcA + 2 * kTcB;
static constexpr size_t kTcCsBytes = (size_t)64 * 128 * 4;  // QKV: the RoPE rows of the chunk's 64 tokens
// only the QKV epilogue keeps RoPE rows: the other launches stay small enough for two CTAs per SM, so one
// CTA's epilogue overlaps the other's k-loop
__host__ __device__ constexpr size_t tc_cs_bytes(int epi) { return epi == EPI_QKV_ROPE ? kTcCsBytes : 0; }
// dynamic shared memory of a TC launch with S K-splits: [ring][RoPE rows][split-K receive buffer] + 1 KB to
// align the ring (the receive buffer is separate: peers push into it while this CTA still runs its ring)
__host__ __device__ inline size_t tc_recv_bytes(int S) { return S > 1 ? (size_t)S * 128 * gemm_kblk(8, S) * 4 : 0; }
__host__ __device__ inline size_t tc_smem(int S, int epi = EPI_QKV_ROPE) {
  return (size_t)kTcStages * kTcStage + tc_cs_bytes(epi) + tc_recv_bytes(S) + 1024;
}

ENG_DEVICE uint8_t* tc_ring(uint8_t* smem) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem) + 1023) & ~static_cast<uintptr_t>(1023));
}

template <int NT, int EPI, bool NORM_IN, bool TC>
ENG_DEVICE void gemm_body(const GemmParams& p, const TcMaps* tm) {
  constexpr int kPre = NT <= 2 ? kPreMax / 2 : (NT == 4 ? kPreMax / 4 : kPreMax / 8);
  constexpr int kUnroll = NT >= 8 ? 2 : 4;  // weight k-tiles loaded per group (register budget)
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float s_rstd[64];
  __shared__ int s_xrow[64];           // row of X of each staged token (x_rows, a step input, or the token)
  __shared__ int s_flag;
  __shared__ int s_slot[64];           // EPI_QKV_ROPE: KV slot of each finished token (-1 padding, -2 bad)
  __shared__ int s_pos[64];            //               and its position
  __shared__ float s_cs[kCsTokens][128];  //          and its RoPE row (cos, sin pairs) for the first tokens
  __shared__ float s_qn[128], s_kn[128];   //          the QK-norm weights
  __shared__ float s_row[128];  // per output row of this CTA: bias (QKV, STORE) or next norm weight (RESID)
  __shared__ __align__(8) uint64_t s_wbar, s_xbar;
  __shared__ __align__(8) uint64_t s_full[TC ? kTcStages : 1], s_empty[TC ? kTcStages : 1], s_done;
  __shared__ uint32_t s_tmem;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rgi = blockIdx.x, split = blockIdx.y, chunk = blockIdx.z;
  const int S = p.S;
  const int n0 = chunk * 64;
  const int KT = p.K >> 5;
  const int ktn = p.kt_per_split;
  const int kt0 = split * ktn;
  const int RG = p.RG, KG = 8 / RG;
  const int rt = warp % RG, kg = warp / RG;
  const int row_tile = rgi * RG + rt;
  const int ntok = min(NT * 8, p.T - n0);  // valid tokens of this chunk
  const GemmSmem sm = gemm_smem(NT, RG, ktn, S);
  const int rows = 16 * RG;
  const int row0 = rgi * rows;

  // ---- before waiting: weights and step inputs do not depend on the preceding kernel
  uint8_t* area = smem + sm.w_bytes;  // X staging, then the reduction tiles
  bf16* xs = reinterpret_cast<bf16*>(area);
  const int xstride = sm.piece * 32 + 8;           // padded row stride of a plane (16-byte multiple)
  bf16* xl = xs + (size_t)NT * 8 * xstride;        // lo plane
  cg::cluster_group cluster = cg::this_cluster();
  const uint4* wp = reinterpret_cast<const uint4*>(p.W) + ((size_t)row_tile * KT + kt0) * 64 + lane;
  const int pn0 = min(sm.piece, ktn);
  uint4 pre[kPre][2];
  const int nk = (p.K >> 6) / S;  // TC: k-blocks of 64 of this split
  const int kb0 = split * nk;      //     starting here
  if constexpr (TC) {
    // tensor memory for the accumulator, the stage barriers, and the weight tiles of the first stages
    if (warp == 0) tmem_alloc<64>(&s_tmem);
    if (threadIdx.x == 0) {
      for (int st = 0; st < kTcStages; ++st) {
        mbar_init(&s_full[st], 1);
        mbar_init(&s_empty[st], 1);
      }
      mbar_init(&s_done, 1);
      uint8_t* ring = tc_ring(smem);
      for (int kb = 0; kb < min(kTcStages, nk); ++kb) {
        mbar_expect_tx(&s_full[kb], kTcStage);
        tma_tile_2d(ring + (size_t)kb * kTcStage, &tm->w, (kb0 + kb) * 64, row0, &s_full[kb]);
      }
    }
  } else if (threadIdx.x == 0) {
    mbar_init(&s_xbar, 1);
    if (sm.tma) {  // the CTA's whole slice (RG row tiles x ktn k-tiles, contiguous per row tile)
      mbar_init(&s_wbar, 1);
      mbar_expect_tx(&s_wbar, (uint32_t)sm.w_bytes);
      for (int r = 0; r < RG; ++r)
        tma_load_1d(smem + (size_t)r * ktn * 1024, p.W + ((size_t)(rgi * RG + r) * KT + kt0) * 512,
                    (uint32_t)ktn * 1024u, &s_wbar);
    }
  }
  if (!TC && !sm.tma) {
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int kt = kg + u * KG;
      if (kt < pn0) {
        pre[u][0] = ld_stream16(wp + (size_t)kt * 64);
        pre[u][1] = ld_stream16(wp + (size_t)kt * 64 + 32);
      } else {
        pre[u][0] = pre[u][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (threadIdx.x < RG && ktn > kPre * KG)
      prefetch_l2(p.W + ((size_t)(rgi * RG + threadIdx.x) * KT + kt0) * 512, (uint32_t)ktn * 1024u);
  }
  if (threadIdx.x == 32 && p.pf_bytes) prefetch_share(p.pf_ptr, p.pf_bytes);
  // padding token rows of both planes are zero (the copies below fill rows < ntok only)
  if constexpr (!TC) {
    const int pad = (NT * 8 - ntok) * xstride / 8;  // 16-byte chunks per plane
    uint4* zh = reinterpret_cast<uint4*>(xs + (size_t)ntok * xstride);
    uint4* zl = reinterpret_cast<uint4*>(xl + (size_t)ntok * xstride);
    for (int i = threadIdx.x; i < pad; i += 256) zh[i] = zl[i] = make_uint4(0u, 0u, 0u, 0u);
  }

  if (threadIdx.x < ntok) s_xrow[threadIdx.x] = p.x_rows ? p.x_rows[n0 + threadIdx.x] : n0 + threadIdx.x;
  // tokens this CTA finishes: a block of kblk from split * kblk (all of them when S == 1)
  const int kblk = S > 1 ? gemm_kblk(NT, S) : NT * 8;
  const int tok_first = S > 1 ? split * kblk : 0;
  const int tok_step = 1;
  const int nown = max(0, min(kblk, ntok - tok_first));
  if (EPI == EPI_QKV_ROPE) {
    // step inputs (positions, lengths, block tables) are final before the step's first kernel: resolve
    // each token's KV slot and fetch its RoPE row while the preceding kernel still runs
    if (threadIdx.x < nown) {
      const int tkn = n0 + tok_first + threadIdx.x * tok_step;
      const int rq = p.tok2req[tkn];
      const int pos = p.positions[tkn];
      int slot = -1;
      if (p.seq_lens[rq] != 0) {
        if (pos < 0 || (pos >> 4) >= p.mbs || pos >= p.max_pos) {
          slot = -2;
        } else {
          const int bb = p.bt[(size_t)rq * p.mbs + (pos >> 4)];
          slot = (bb < 0 || bb >= p.NB) ? -3 : bb * 16 + (pos & 15);
        }
      }
      s_slot[threadIdx.x] = slot;
      s_pos[threadIdx.x] = (pos < 0 || pos >= p.max_pos) ? 0 : pos;
    }
    __syncthreads();
    if constexpr (TC) {  // every owned token's RoPE row, copied asynchronously (landed before the epilogue)
      float* cs_tab = reinterpret_cast<float*>(tc_ring(smem) + (size_t)kTcStages * kTcStage);
      const int q4 = p.d / 4;
      for (int i = threadIdx.x; i < nown * q4; i += 256) {
        const int k = i / q4, c = i - k * q4;
        cp_async16(cs_tab + (size_t)k * p.d + c * 4, p.cos_sin + (size_t)s_pos[k] * p.d + c * 4);
      }
      cp_async_commit();
    } else {
      for (int i = threadIdx.x; i < min(nown, kCsTokens) * p.d; i += 256) {
        const int k = i / p.d, j = i - k * p.d;
        s_cs[k][j] = p.cos_sin[(size_t)s_pos[k] * p.d + j];
      }
    }
    if (threadIdx.x < p.d) {
      s_qn[threadIdx.x] = p.q_norm ? p.q_norm[threadIdx.x] : 1.f;
      s_kn[threadIdx.x] = p.k_norm ? p.k_norm[threadIdx.x] : 1.f;
    }
  }
  if (threadIdx.x < rows) {
    const float* rv = EPI == EPI_RESID ? p.next_norm_w : p.bias;
    s_row[threadIdx.x] = rv ? rv[row0 + threadIdx.x] : (EPI == EPI_RESID ? 1.f : 0.f);
  }
  if constexpr (TC) tc_fence_before();
  __syncthreads();        // barriers initialised, padding rows zeroed (TC: tensor memory allocated)
  if constexpr (TC) tc_fence_after();
  if (S > 1) cluster.sync();  // every CTA of the cluster has started before any pushes into its memory
  // The next kernel may launch (and start its own early copies) only once this kernel's inputs have
  // arrived (see the trigger below): its early copies would otherwise queue ahead of these critical loads.
  pdl_wait();

  // X piece [pc, pc + pn) k-tiles.  A few token rows: one bulk copy per row and plane, issued by warp 0.
  // More rows: the CTA's threads issue 16-byte asynchronous copies (bulk copies are issued one after
  // another, and dozens of them take microseconds to issue).
  const bool x_async = ntok > 4;
  auto issue_x = [&](int pc, int pn) {
    if (x_async) {
      const int cpr = pn * 4;  // 16-byte chunks of a row in one plane
      if (cpr >= 16) {         // a warp per token row, lanes over its chunks
        for (int r = warp; r < ntok; r += 8) {
          const size_t off = (size_t)s_xrow[r] * p.ldx + (size_t)(kt0 + pc) * 32;
          bf16* dh = xs + (size_t)r * xstride;
          bf16* dl = xl + (size_t)r * xstride;
          for (int c = lane; c < cpr; c += 32) {
            cp_async16(dh + c * 8, p.Xh + off + c * 8);
            cp_async16(dl + c * 8, p.Xl + off + c * 8);
          }
        }
      } else {
        for (int i = threadIdx.x; i < 2 * ntok * cpr; i += 256) {
          const int plane = i >= ntok * cpr;
          const int rem = i - plane * ntok * cpr, r = rem / cpr, c = rem - r * cpr;
          const size_t off = (size_t)s_xrow[r] * p.ldx + (size_t)(kt0 + pc) * 32 + c * 8;
          cp_async16((plane ? xl : xs) + (size_t)r * xstride + c * 8, (plane ? p.Xl : p.Xh) + off);
        }
      }
      cp_async_commit();
    } else if (warp == 0) {
      if (lane == 0) mbar_expect_tx(&s_xbar, (uint32_t)(ntok * pn * 64 * 2));
      __syncwarp();
      for (int r = lane; r < ntok; r += 32) {
        const size_t off = (size_t)s_xrow[r] * p.ldx + (size_t)(kt0 + pc) * 32;
        tma_load_1d(xs + (size_t)r * xstride, p.Xh + off, (uint32_t)pn * 64u, &s_xbar);
        tma_load_1d(xl + (size_t)r * xstride, p.Xl + off, (uint32_t)pn * 64u, &s_xbar);
      }
    }
  };
  if constexpr (TC) {
    if (threadIdx.x == 0) {  // the activation tiles of the first stages
      uint8_t* ring = tc_ring(smem);
      for (int kb = 0; kb < min(kTcStages, nk); ++kb) {
        tma_tile_2d(ring + (size_t)kb * kTcStage + kTcA, &tm->xh, (kb0 + kb) * 64, n0, &s_full[kb]);
        tma_tile_2d(ring + (size_t)kb * kTcStage + kTcA + kTcB, &tm->xl, (kb0 + kb) * 64, n0, &s_full[kb]);
      }
    }
  } else {
    issue_x(0, pn0);
  }

  // EPI_RESID: the residual values this thread updates in the epilogue (warps over its first two owned
  // tokens, lanes over up to four rows each), fetched now so the epilogue needs no further round trip
  constexpr int kOldTok = TC ? 8 : 2;  // owned tokens per warp whose residual values are fetched here
  float h_old[kOldTok][4];
  if (EPI == EPI_RESID) {
#pragma unroll
    for (int a = 0; a < kOldTok; ++a) {
      const int k = warp + 8 * a;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int r = lane + 32 * b;
        h_old[a][b] = (k < nown && r < rows) ? p.resid[(size_t)(n0 + tok_first + k * tok_step) * p.N + row0 + r] : 0.f;
      }
    }
  }
  if (NORM_IN) {  // 1 / rms of each staged token, from its producer's partial sums of squares (a warp per
                  // token; every load of the warp's tokens issued before the first reduction)
    float part_ss[NT];
#pragma unroll
    for (int a = 0; a < NT; ++a) {
      const int r = warp + 8 * a;
      float ss = 0.f;
      if (r < ntok) {  // the first 32 parts with no loop, so that every token's load is issued at once
        const float* part = p.sq_in + (size_t)s_xrow[r] * p.sq_stride;
        ss = lane < p.sq_parts ? part[lane] : 0.f;
        for (int j = lane + 32; j < p.sq_parts; j += 32) ss += part[j];
      }
      part_ss[a] = ss;
    }
#pragma unroll
    for (int a = 0; a < NT; ++a) {
      const int r = warp + 8 * a;
      const float ss = warp_sum(part_ss[a]);
      if (lane == 0 && r < ntok) s_rstd[r] = rsqrtf(ss / (float)p.K + p.eps);
    }
  }

  float* ts;
  constexpr int TS = NT * 8 + 1;  // token stride (padded)
  if constexpr (!TC) {
    float acc[NT][4], accl[NT][4];
  #pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      accl[nt][0] = accl[nt][1] = accl[nt][2] = accl[nt][3] = 0.f;
    }

    const uint4* ws = reinterpret_cast<const uint4*>(smem) + (size_t)rt * ktn * 64 + lane;  // tma: this warp's row tile
    if (sm.tma && !mbar_wait(&s_wbar, 0, 1u << 26)) {
      set_status(p.status, ST_TIMEOUT);
      mbar_wait(&s_wbar, 0, 1u << 26);  // never leave while the copy may still write shared memory
    }
    int piece_no = 0;
    for (int pc = 0; pc < ktn; pc += sm.piece, ++piece_no) {
      const int pn = min(sm.piece, ktn - pc);
      if (pc > 0) {  // every warp is done with the previous piece before its rows are overwritten
        __syncthreads();
        if (warp == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_x(pc, pn);
      }
      if (x_async) {
        cp_async_wait<0>();
        __syncthreads();
      } else if (!mbar_wait(&s_xbar, piece_no & 1, 1u << 26)) {
        set_status(p.status, ST_TIMEOUT);
        mbar_wait(&s_xbar, piece_no & 1, 1u << 26);
      }
      if (piece_no == 0) pdl_trigger();  // inputs in: the next kernel may launch

      if (sm.tma) {
        constexpr int UT = kUnroll;
        for (int base = kg; base < pn; base += KG * UT) {
          uint4 a[UT][2];
  #pragma unroll
          for (int u = 0; u < UT; ++u) {
            const int kt = base + u * KG;
            if (kt < pn) {
              a[u][0] = ws[(size_t)(pc + kt) * 64];
              a[u][1] = ws[(size_t)(pc + kt) * 64 + 32];
            }
          }
  #pragma unroll
          for (int u = 0; u < UT; ++u) {
            const int kt = base + u * KG;
            if (kt < pn) mma_tile<NT>(acc, accl, a[u][0], a[u][1], xs, xl, xstride, kt, lane);
          }
        }
        continue;
      }
      int first = kg;
      if (pc == 0) {  // the fragments loaded before waiting
  #pragma unroll
        for (int u = 0; u < kPre; ++u) {
          const int kt = kg + u * KG;
          if (kt < pn) mma_tile<NT>(acc, accl, pre[u][0], pre[u][1], xs, xl, xstride, kt, lane);
        }
        first = kg + kPre * KG;
      }
      constexpr int U = kUnroll;
      for (int base = first; base < pn; base += KG * U) {
        uint4 a[U][2];
  #pragma unroll
        for (int u = 0; u < U; ++u) {
          const int kt = base + u * KG;
          if (kt < pn) {
            a[u][0] = ld_stream16(wp + (size_t)(pc + kt) * 64);
            a[u][1] = ld_stream16(wp + (size_t)(pc + kt) * 64 + 32);
          } else {
            a[u][0] = a[u][1] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
  #pragma unroll
        for (int u = 0; u < U; ++u) {
          const int kt = base + u * KG;
          if (kt < pn) mma_tile<NT>(acc, accl, a[u][0], a[u][1], xs, xl, xstride, kt, lane);
        }
      }
    }
  #pragma unroll
    for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
      for (int j = 0; j < 4; ++j) acc[nt][j] += accl[nt][j];

    // ---- this CTA's tile: sum the KG warps of each row tile in warp order
    __syncthreads();
    float4* red = reinterpret_cast<float4*>(area);
    ts = reinterpret_cast<float*>(area + sm.red_bytes);
    if (KG == 1) {  // one warp per row tile: its fragments go straight into the tile
  #pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r0 = rt * 16 + (lane >> 2), c0 = nt * 8 + 2 * (lane & 3);
        ts[r0 * TS + c0] = acc[nt][0];
        ts[r0 * TS + c0 + 1] = acc[nt][1];
        ts[(r0 + 8) * TS + c0] = acc[nt][2];
        ts[(r0 + 8) * TS + c0 + 1] = acc[nt][3];
      }
    } else {
  #pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        red[(warp * NT + nt) * 32 + lane] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
      __syncthreads();
    }
    for (int i = threadIdx.x; KG > 1 && i < RG * NT * 32; i += 256) {
      const int ln = i & 31, nt = (i >> 5) % NT, r_t = (i >> 5) / NT;
      float4 v = red[((0 * RG + r_t) * NT + nt) * 32 + ln];
      for (int j = 1; j < KG; ++j) {
        const float4 w = red[((j * RG + r_t) * NT + nt) * 32 + ln];
        v.x += w.x;
        v.y += w.y;
        v.z += w.z;
        v.w += w.w;
      }
      const int r0 = r_t * 16 + (ln >> 2), c0 = nt * 8 + 2 * (ln & 3);
      ts[r0 * TS + c0] = v.x;
      ts[r0 * TS + c0 + 1] = v.y;
      ts[(r0 + 8) * TS + c0] = v.z;
      ts[(r0 + 8) * TS + c0 + 1] = v.w;
    }
    __syncthreads();

  } else {
    // ---- tensor-core path: one thread issues every k-block's MMAs as its stage lands and refills the stage
    // the previous k-block used once those MMAs are done
    uint8_t* ring = tc_ring(smem);
    pdl_trigger();  // the first stages' copies are in flight: the next kernel may launch
    // lane 0 of warp 0 issues; the rest of warp 0 waits at the warp barrier below, not on an mbarrier, so
    // the issuing lane never shares its warp with lanes that spin
    if (warp == 0 && lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(128, 64);
      int issued = min(kTcStages, nk);  // k-blocks whose copies were issued
      int kb = 0;
      for (; kb < nk; ++kb) {
        const int st = kb % kTcStages;
        uint8_t* stage = ring + (size_t)st * kTcStage;
        if (!mbar_wait(&s_full[st], (kb / kTcStages) & 1, 1u << 26)) {
          set_status(p.status, ST_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint64_t ad = umma_desc_sw128(stage), bh = umma_desc_sw128(stage + kTcA),
                       bl = umma_desc_sw128(stage + kTcA + kTcB);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          umma_bf16(s_tmem, ad + 2 * k, bh + 2 * k, idesc, (kb | k) != 0);
          umma_bf16(s_tmem, ad + 2 * k, bl + 2 * k, idesc, 1u);
        }
        umma_commit(&s_empty[st]);
        const int pk = kb - 1, nkb = pk + kTcStages;
        if (pk >= 0 && nkb < nk) {
          const int ps = pk % kTcStages;
          if (!mbar_wait(&s_empty[ps], (pk / kTcStages) & 1, 1u << 26)) {
            set_status(p.status, ST_TIMEOUT);
            ++kb;
            break;
          }
          uint8_t* pst = ring + (size_t)ps * kTcStage;
          mbar_expect_tx(&s_full[ps], kTcStage);
          tma_tile_2d(pst, &tm->w, (kb0 + nkb) * 64, row0, &s_full[ps]);
          tma_tile_2d(pst + kTcA, &tm->xh, (kb0 + nkb) * 64, n0, &s_full[ps]);
          tma_tile_2d(pst + kTcA + kTcB, &tm->xl, (kb0 + nkb) * 64, n0, &s_full[ps]);
          issued = nkb + 1;
        }
      }
      // after a timeout, copies still in flight land before the ring is reused or the CTA exits
      for (int q = kb; q < issued; ++q) mbar_wait(&s_full[q % kTcStages], (q / kTcStages) & 1, 1u << 26);
      umma_commit(&s_done);
    }
    if (warp == 0) __syncwarp();
    if (!mbar_wait(&s_done, 0, 1u << 26)) {
      set_status(p.status, ST_TIMEOUT);
      mbar_wait(&s_done, 0, 1u << 26);
    }
    tc_fence_after();
    // warp w reads its TMEM lane quarter (rows 32 (w % 4) ..) and column half (tokens 32 (w / 4) ..)
    ts = reinterpret_cast<float*>(ring);
    {
      float v[32];
      tmem_ld32(s_tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)((warp >> 2) * 32), v);
      const int r = (warp & 3) * 32 + lane;
#pragma unroll
      for (int j = 0; j < 32; ++j) ts[r * TS + (warp >> 2) * 32 + j] = v[j];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free<64>(s_tmem);
    if (EPI == EPI_QKV_ROPE) {  // the RoPE rows copied before the wait
      cp_async_wait<0>();
      __syncthreads();
    }
  }
  // ---- split-K across the cluster: CTA `split` finishes its block of tokens (sums in split order)
  if (S > 1) {
    // push this CTA's partial sums of the tokens CTA q finishes into q's receive buffer (4 tokens per
    // 16-byte store), then every CTA adds its block's partials in split order (its own at its position)
    float* recv = TC ? reinterpret_cast<float*>(tc_ring(smem) + (size_t)kTcStages * kTcStage + tc_cs_bytes(EPI))
                    : reinterpret_cast<float*>(area + sm.recv_off);  // [S][rows][kblk]
    const int groups = kblk / 4;
    for (int i = threadIdx.x; i < S * rows * groups; i += 256) {
      const int q = i / (rows * groups), rem = i - q * rows * groups;
      const int r = rem / groups, c = rem - r * groups;
      const int t0 = q * kblk + 4 * c;
      if (q == split || t0 >= ntok) continue;
      const float* src = ts + r * TS + t0;
      const float4 v = make_float4(src[0], t0 + 1 < ntok ? src[1] : 0.f, t0 + 2 < ntok ? src[2] : 0.f,
                                   t0 + 3 < ntok ? src[3] : 0.f);
      *reinterpret_cast<float4*>(cluster.map_shared_rank(recv, q) + ((size_t)split * rows + r) * kblk + 4 * c) = v;
    }
    cluster.sync();
    // lanes over a row's tokens (2^ksh >= nown lanes a row), 32 >> ksh rows a warp pass
    const int ksh = nown <= 1 ? 0 : 32 - __clz(nown - 1);
    if (ksh <= 5) {
      for (int r = (warp << (5 - ksh)) + (lane >> ksh); r < rows; r += 8 << (5 - ksh)) {
        const int k = lane & ((1 << ksh) - 1);
        if (k >= nown) continue;
        const int tok = tok_first + k;
        float v = 0.f;
        for (int sp = 0; sp < S; ++sp) v += sp == split ? ts[r * TS + tok] : recv[((size_t)sp * rows + r) * kblk + k];
        ts[r * TS + tok] = v;
      }
    } else {
      for (int i = threadIdx.x; i < rows * nown; i += 256) {
        const int r = i / nown, k = i - r * nown;
        const int tok = tok_first + k;
        float v = 0.f;
        for (int sp = 0; sp < S; ++sp) v += sp == split ? ts[r * TS + tok] : recv[((size_t)sp * rows + r) * kblk + k];
        ts[r * TS + tok] = v;
      }
    }
    __syncthreads();
  }
  // RMSNorm(h) W^T = (1 / rms(h)) ((h * w) W^T): with NORM_IN every epilogue scales token tok's sums by
  // rstd(tok) as it reads them.  rows (16 RG) is a power of two.
  auto rstd = [&](int tok) { return NORM_IN ? s_rstd[tok] : 1.f; };
  const int rows_sh = __ffs(rows) - 1;
  if (EPI == EPI_STORE_F32) {
    for (int i = threadIdx.x; i < rows * nown; i += 256) {
      const int k = i >> rows_sh, r = i & (rows - 1);
      const int tok = tok_first + k * tok_step;
      p.out_f32[(size_t)(n0 + tok) * p.ldo + row0 + r] = ts[r * TS + tok] * rstd(tok) + s_row[r];
    }
  } else if (EPI == EPI_RESID) {
    // h += Y, this CTA's share of each token's sum of squares (lanes over rows, warps over tokens) and
    // the next GEMM's operand planes of h * next norm weight
    for (int k = warp; k < nown; k += 8) {
      const int tok = tok_first + k * tok_step;
      const size_t base = (size_t)(n0 + tok) * p.N + row0;
      float* hrow = p.resid + base;
      float ss = 0.f;
      for (int r = lane; r < rows; r += 32) {
        const int a = k >> 3, b = r >> 5;
        const float old = (a < kOldTok && b < 4) ? h_old[a % kOldTok][b & 3] : hrow[r];
        const float v = old + ts[r * TS + tok];
        hrow[r] = v;
        put_split(p.xh_out, p.xl_out, base + r, v * s_row[r]);
        ss += v * v;
      }
      ss = warp_sum(ss);
      if (lane == 0) p.sq_out[(size_t)(n0 + tok) * p.sq_stride + rgi] = ss;
    }
  } else if (EPI == EPI_SILU) {
    const int I = p.N >> 1;
    const int half = rows >> 1;  // gate rows j: tile row r < 8 of each 16-row tile; up rows: r + 8
    for (int i = threadIdx.x; i < half * nown; i += 256) {
      const int k = i >> (rows_sh - 1), jj = i & (half - 1);
      const int tok = tok_first + k * tok_step;
      const int r = (jj >> 3) * 16 + (jj & 7);
      const float rs = rstd(tok);
      const float ga = ts[r * TS + tok] * rs, up = ts[(r + 8) * TS + tok] * rs;
      put_split(p.xh_out, p.xl_out, (size_t)(n0 + tok) * I + (row0 >> 1) + jj, ga / (1.f + expf(-ga)) * up);
    }
  } else if (EPI == EPI_QKV_ROPE) {
    const int D = p.d;
    const int E = D / 32;  // 2 or 4 elements of a head per lane (loops below unrolled to 4)
    const int nheads_cta = rows / D;
    for (int item = warp; item < nown * nheads_cta; item += 8) {
      const int k = item / nheads_cta, hc = item - k * nheads_cta;
      const int tok = tok_first + k * tok_step;
      const int head = (row0 / D) + hc;
      const int tkn = n0 + tok;
      const int rbase = hc * D;
      const int slot = s_slot[k];
      int blk = p.NB, off = 0;
      if (slot >= 0) {
        blk = slot >> 4;
        off = slot & 15;
      }
      if (head == 0 && lane == 0) {
        p.slots[tkn] = slot >= 0 ? slot : -1;
        if (slot < -1) set_status(p.status, slot == -2 ? ST_BAD_POSITION : ST_BAD_BLOCK);
      }
      float x[4];
      const float rs_in = rstd(tok);
      _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) {
        const int r = rbase + lane * E + e;
        x[e] = ts[r * TS + tok] * rs_in + s_row[r];
      }
      const bool is_q = head < p.Hq;
      const bool is_k = !is_q && head < p.Hq + p.Hkv;
      if (is_q || is_k) {
        const float* nw = is_q ? s_qn : s_kn;
        if (is_q ? p.q_norm != nullptr : p.k_norm != nullptr) {
          float ss = 0.f;
          _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) ss += x[e] * x[e];
          ss = warp_sum(ss);
          const float rs = rsqrtf(ss / (float)D + p.eps);
          _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) x[e] = x[e] * rs * nw[lane * E + e];
        }
        // rotate-half RoPE: element i < D/2 pairs with i + D/2, held by lane ^ 16
        const float* cs = TC ? reinterpret_cast<const float*>(tc_ring(smem) + (size_t)kTcStages * kTcStage) + (size_t)k * D
                             : (k < kCsTokens ? s_cs[k] : p.cos_sin + (size_t)s_pos[k] * D);  // [D/2][2]
        float y[4];
        _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) {
          const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
          const int ii = (lane & 15) * E + e;
          const float c = cs[2 * ii], sn = cs[2 * ii + 1];
          y[e] = (lane < 16) ? (x[e] * c - other * sn) : (x[e] * c + other * sn);
        }
        _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) x[e] = y[e];
      }
      if (is_q) {  // q stays fp32: the attention splits it into hi/lo operands
        float* dq = p.q_out + ((size_t)tkn * p.Hq + head) * D + lane * E;
        _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) dq[e] = x[e];
      } else {     // the cache holds bf16
        const int kvh = is_k ? head - p.Hq : head - p.Hq - p.Hkv;
        bf16* plane = is_k ? p.k_pool : p.v_pool;
        bf16* dst = plane + (((size_t)blk * p.Hkv + kvh) * 16 + off) * D;
        _Pragma("unroll") for (int e = 0; e < 4; e += 2) if (e < E)
          *reinterpret_cast<uint32_t*>(dst + lane * E + e) = pack_bf16x2(x[e], x[e + 1]);
      }
    }
  } else if (EPI == EPI_LMHEAD) {
    const bool wl = *p.write_logits != 0;
    const bool wk = wl && p.keys_out && *p.write_keys != 0, we = wl && p.row_ext;  // (uniform)
    const uint32_t rng[4] = {p.rng[0], p.rng[1], p.rng[2], p.rng[3]};
    for (int k = warp; k < nown; k += 8) {
      const int tok = tok_first + k * tok_step;
      const int tkn = n0 + tok;
      const float it = p.inv_temp[tkn];
      const float rs_in = rstd(tok);
      unsigned long long best = 0ull;
      uint32_t omax = 0u, omin_inv = 0u;  // extremes of the finite logits, as order-preserving bits
      for (int r = lane; r < rows; r += 32) {
        const int v = row0 + r;
        const float z = ts[r * TS + tok] * rs_in;
        if (wl) p.logits[(size_t)tkn * p.N + v] = z;
        const float key = sample_key(z, it, rng, (uint32_t)tkn, (uint32_t)v);
        if (wk) p.keys_out[(size_t)tkn * p.N + v] = key;
        if (we && (__float_as_uint(z) & 0x7F800000u) != 0x7F800000u) {
          uint32_t f = __float_as_uint(z);
          if (f == 0x80000000u) f = 0u;  // -0 orders as +0
          const uint32_t o = (f & 0x80000000u) ? ~f : (f | 0x80000000u);
          omax = o > omax ? o : omax;
          omin_inv = ~o > omin_inv ? ~o : omin_inv;
        }
        if (key != key) {
          set_status(p.status, ST_NAN);
        } else {
          const unsigned long long pk = pack_key_index(key, (uint32_t)v);
          best = pk > best ? pk : best;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, o);
        best = x > best ? x : best;
      }
      if (lane == 0 && best) atomicMax(p.best + tkn, best);
      if (we) {
        omax = __reduce_max_sync(0xffffffffu, omax);
        omin_inv = __reduce_max_sync(0xffffffffu, omin_inv);
        if (lane == 0 && omax) {
          atomicMax(p.row_ext + 2 * tkn, omax);
          atomicMax(p.row_ext + 2 * tkn + 1, omin_inv);
        }
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int total = gridDim.x * gridDim.y * gridDim.z;
      const int old = atomicAdd(p.done_counter, 1);
      s_flag = (old == total - 1);
    }
    __syncthreads();
    if (s_flag) {
      __threadfence();
      for (int r = threadIdx.x; r < p.T; r += blockDim.x) {
        const unsigned long long b = atomicExch(p.best + r, 0ull);
        p.out_ids[r] = (int)unpack_index(b);
      }
      if (threadIdx.x == 0) *p.done_counter = 0;
    }
  }
}

// Warp-MMA path (decode sizes and the LM head).
template <int NT, int EPI, bool NORM_IN>
__global__ void __launch_bounds__(256, 2) k_gemm(GemmParams p) {
  gemm_body<NT, EPI, NORM_IN, false>(p, nullptr);
}

// Tensor-core path (steps of kTcTokens tokens or more).
template <int EPI, bool NORM_IN>
__global__ void __launch_bounds__(256, 1) k_gemm_tc(GemmParams p, const __grid_constant__ TcMaps tm) {
  gemm_body<8, EPI, NORM_IN, true>(p, &tm);
}

// ------------------------------------------------------------------ host side

static constexpr int kMaxCluster = 8;

void gemm_plan(int N, int K, int rg_fixed, int sms, int* RG, int* S, int* kt_per_split) {
  // Every round trip after the kernel's wait costs about a microsecond, and so does a cluster reduction,
  // so the plan first looks for the fewest K splits whose per-CTA weight slice still fits the shared-memory
  // budget of the bulk copy (the slice is then fetched before the wait), with at most one wave of CTAs at
  // one CTA per SM (the other half of the SM stays free for the next kernel's early CTAs); among those it
  // takes the most CTAs.  When no slice fits, it takes the most CTAs in one wave (ties: fewer splits).
  const int tiles = N / 16, KT = K / 32;
  const int wave = sms;
  int best_rg = 0, best_s = 0, best_ctas = 0;
  for (int sp = 1; sp <= kMaxCluster && sp <= KT && best_ctas == 0; ++sp) {
    if (KT % sp) continue;
    for (int rg = 1; rg <= 8; rg <<= 1) {
      if ((rg_fixed > 0 && rg != rg_fixed) || tiles % rg) continue;
      const int ctas = tiles / rg * sp;
      if (ctas > wave || (size_t)rg * (KT / sp) * 1024 > kTmaMaxBytes) continue;
      if (ctas > best_ctas) {
        best_ctas = ctas;
        best_rg = rg;
        best_s = sp;
      }
    }
  }
  if (best_ctas == 0) {
    for (int rg = 1; rg <= 8; rg <<= 1) {
      if ((rg_fixed > 0 && rg != rg_fixed) || tiles % rg) continue;
      for (int sp = 1; sp <= kMaxCluster && sp <= KT; ++sp) {
        if (KT % sp) continue;
        const int ctas = tiles / rg * sp;
        if (ctas > wave) continue;
        if (ctas > best_ctas || (ctas == best_ctas && sp < best_s)) {
          best_ctas = ctas;
          best_rg = rg;
          best_s = sp;
        }
      }
    }
  }
  if (best_ctas == 0) {  // more row tiles than one wave holds: the largest tiles, no split
    best_rg = rg_fixed > 0 ? rg_fixed : 8;
    while (best_rg > 1 && tiles % best_rg) best_rg >>= 1;
    best_s = 1;
  }
  *RG = best_rg;
  *S = best_s;
  *kt_per_split = KT / best_s;
}

void gemm_plan_large(int N, int K, int rg_fixed, int sms, int* RG, int* S, int* kt_per_split) {
  // Steps of more than 8 tokens: every CTA also reads its K-range of the activation planes for each token
  // (T x K-range x 4 bytes from L2), which at 32 tokens outweighs a thin weight slice.  The plan minimises
  // the bytes one SM moves, waves x (2 W + X) with W the CTA's weight slice (from HBM, counted twice) and X
  // its activation slice for 32 tokens, over row groups of 1..8 tiles and 1..8 K splits in at most two
  // waves (ties: fewer CTAs, then fewer splits).  Falls back to the small-step plan when nothing fits.
  const int tiles = N / 16, KT = K / 32;
  const int wave = sms;
  double best = 0.0;
  int best_rg = 0, best_s = 0, best_ctas = 0;
  for (int rg = 1; rg <= 8; rg <<= 1) {
    if ((rg_fixed > 0 && rg != rg_fixed) || tiles % rg) continue;
    for (int sp = 1; sp <= kMaxCluster && sp <= KT; ++sp) {
      if (KT % sp) continue;
      const int ctas = tiles / rg * sp;
      if (ctas > 2 * wave) continue;
      const double w = (double)rg * 16 * (K / sp) * 2, x = 32.0 * (K / sp) * 4;
      const double cost = (double)((ctas + wave - 1) / wave) * (2.0 * w + x);
      if (best_ctas == 0 || cost < best || (cost == best && (ctas < best_ctas || (ctas == best_ctas && sp < best_s)))) {
        best = cost;
        best_rg = rg;
        best_s = sp;
        best_ctas = ctas;
      }
    }
  }
  if (best_ctas == 0) {
    gemm_plan(N, K, rg_fixed, sms, RG, S, kt_per_split);
    return;
  }
  *RG = best_rg;
  *S = best_s;
  *kt_per_split = KT / best_s;
}

template <int NT, int EPI, bool NORM_IN, bool TC>
static cudaError_t launch_nt(const GemmParams& p, const LaunchOpts& o, cudaStream_t s, dim3 grid, const TcMaps* tm) {
  const size_t smem_bytes = TC ? tc_smem(p.S, EPI) : gemm_smem(NT, p.RG, p.kt_per_split, p.S).total;
  cudaError_t ae;
  if constexpr (TC)
    ae = ensure_smem_limit(reinterpret_cast<const void*>(k_gemm_tc<EPI, NORM_IN>), (int)kSmemBudget);
  else
    ae = ensure_smem_limit(reinterpret_cast<const void*>(k_gemm<NT, EPI, NORM_IN>), (int)kSmemBudgetMma);
  if (ae != cudaSuccess) return ae;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = o.pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = p.S;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.S > 1 ? 2 : 1;
  if constexpr (TC) return cudaLaunchKernelEx(&cfg, k_gemm_tc<EPI, NORM_IN>, p, *tm);
  else return cudaLaunchKernelEx(&cfg, k_gemm<NT, EPI, NORM_IN>, p);
}

static int chunks_of(int T) { return (T + 63) / 64; }

template <int EPI, bool NORM_IN>
static cudaError_t launch_epi(const GemmParams& p, const LaunchOpts& o, cudaStream_t s, const TcMaps* tc) {
  const int nRG = p.N / 16 / p.RG;
  const dim3 grid(nRG, p.S, chunks_of(p.T));
  if (tc) {
    if (EPI == EPI_LMHEAD || p.RG != 8 || p.x_rows || p.N % 128 || p.K % 64 || (p.K / 64) % p.S ||
        tc_smem(p.S) > kSmemBudget)
      return cudaErrorInvalidValue;
    if constexpr (EPI == EPI_LMHEAD) return cudaErrorInvalidValue;
    else return launch_nt<8, EPI, NORM_IN, true>(p, o, s, grid, tc);
  }
  const int ntiles = p.T >= 64 ? 8 : (p.T + 7) / 8;
  if (ntiles <= 1) return launch_nt<1, EPI, NORM_IN, false>(p, o, s, grid, nullptr);
  if (ntiles <= 2) return launch_nt<2, EPI, NORM_IN, false>(p, o, s, grid, nullptr);
  if (ntiles <= 4) return launch_nt<4, EPI, NORM_IN, false>(p, o, s, grid, nullptr);
  return launch_nt<8, EPI, NORM_IN, false>(p, o, s, grid, nullptr);
}

cudaError_t launch_gemm(const GemmParams& p, int epi, bool norm_in, const LaunchOpts& o, cudaStream_t s,
                        const TcMaps* tc) {
  if (p.T <= 0) return cudaSuccess;
  if (p.S < 1 || p.S > kMaxCluster) return cudaErrorInvalidValue;
  if (norm_in) {
    switch (epi) {
      case EPI_QKV_ROPE: return launch_epi<EPI_QKV_ROPE, true>(p, o, s, tc);
      case EPI_SILU: return launch_epi<EPI_SILU, true>(p, o, s, tc);
      case EPI_LMHEAD: return launch_epi<EPI_LMHEAD, true>(p, o, s, nullptr);
      case EPI_STORE_F32: return launch_epi<EPI_STORE_F32, true>(p, o, s, tc);
    }
  } else {
    switch (epi) {
      case EPI_RESID: return launch_epi<EPI_RESID, false>(p, o, s, tc);
      case EPI_STORE_F32: return launch_epi<EPI_STORE_F32, false>(p, o, s, tc);
    }
  }
  return cudaErrorInvalidValue;
}

bool gemm_slice_fits(int RG, int ktn) { return (size_t)RG * ktn * 1024 <= kTmaMaxBytes; }

bool tc_split_fits(int S) { return S >= 1 && S <= kMaxCluster && tc_smem(S) <= kSmemBudget; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_tc_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  static EncodeTiledFn enc = nullptr;
  if (!enc) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    enc = reinterpret_cast<EncodeTiledFn>(fn);
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

ENG_ELEM_NS_END
}  // namespace grd
