// decode_step.cu -- every layer of a small decode step in one persistent kernel.
//
// At a handful of tokens a decode step moves the model's weights once and does almost no arithmetic, so
// what bounds it is latency: "19. Fast decode", section "Where the time goes", counts the step's small
// kernels, and "One forward per step", section "Bottleneck", finds the step's fixed per-kernel cost larger
// than its weight read.  Graph replay ("33. Removing overhead", section "CUDA graphs for a changing
// batch") removes the host's launch cost but not the device's: each dependent kernel still drains and
// refills the GPU.  This kernel keeps one CTA on every SM for the whole layer stack instead:
//
//   * The work of a layer is five phases -- the fused QKV projection, attention, the output projection
//     with the residual add, the gate|up projection with SiLU-and-mul, the down projection with the
//     residual add.  A static schedule (built on the host per token count) gives every CTA its items of
//     each phase: 16-row tiles of the phase's weight, or one (row, KV head, key split) of attention.
//   * Weights and cached K/V do not depend on the step's activations.  A producer warp walks the CTA's
//     items of every layer in order and streams their weight tiles and K/V blocks into a ring of 32 KB
//     shared-memory slots with bulk copies, as far ahead as the ring allows; the consumer warps only
//     wait for a phase's input activations.
//   * Activations move between phases as 64-bit words: the fp32 value and a 32-bit tag (this step's
//     epoch and the phase), written with one 64-bit store.  A consumer polls the words it needs until
//     every tag matches, so one round trip brings both the data and the signal that it is there.
//     Every reader of a buffer contributes, through the phase chain, to the buffer's next writer, so a
//     word is never overwritten before all its readers have taken it.
//   * RMSNorm: the consumer of h reads the whole row anyway and computes 1 / rms itself (fixed order),
//     so RMSNorm(h) W^T = (1 / rms(h)) ((h * w) W^T) costs nothing extra.  QK-norm and RoPE run in the
//     attention item that reads the head (fp32), before the new K/V are written to the paged pool.
//   * Products run on the tensor cores (m16n8k16, bf16 weights and bf16 hi/lo activation pairs, fp32
//     accumulators, common.cuh), with each warp taking every 8th k-tile and the warps summed in order;
//     attention splits merge in split order.  Results therefore do not depend on the token count, the
//     schedule, or which CTA finishes first: eager steps and graph replays agree bit for bit.
//   * Every wait is bounded: a wait that exceeds the timeout marks the step as given up (one word), sets
//     the status bit, and every other wait of the step then ends at once; copies still in flight are
//     waited for before a CTA exits.
#include "common.cuh"
#include "kernels.h"

namespace grd {

// Seven consumer warps and one producer warp: eight warps (two groups of four) leave a thread up to 255
// registers, where a ninth warp would cap it at 168.
static constexpr int kDsWarps = 7;
static constexpr int kDsConsumers = 32 * kDsWarps;
static constexpr int kDsThreads = kDsConsumers + 32;
static constexpr int kDsMaxSlots = 8;
static constexpr unsigned long long kDsTimeoutNs = 200ull * 1000 * 1000;
static constexpr int kTsStride = 9;  // padded token stride of the 16 x 8 result tile

ENG_DEVICE uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
ENG_DEVICE unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
ENG_DEVICE void ll_store(unsigned long long* p, float v, uint32_t tag) {
  const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// Polling loads carry no compiler memory barrier: what they return is its own signal, and independent
// loads (norm weights, RoPE rows) may be issued alongside them.
ENG_DEVICE void ll_load2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}
ENG_DEVICE unsigned long long ll_load1(const unsigned long long* p) {
  unsigned long long a;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(a) : "l"(p));
  return a;
}
ENG_DEVICE uint32_t ll_tag(unsigned long long w) { return (uint32_t)(w >> 32); }
ENG_DEVICE float ll_val(unsigned long long w) { return __uint_as_float((uint32_t)w); }

// Consumer-only barriers (named barrier 1 over the 256 consumer threads).
ENG_DEVICE void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kDsConsumers) : "memory"); }
ENG_DEVICE int csync_and(int v) {
  int r;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %1, 0;\n bar.red.and.pred p, 1, %2, p;\n selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(v), "n"(kDsConsumers)
      : "memory");
  return r;
}
ENG_DEVICE bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
ENG_DEVICE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
ENG_DEVICE void ldmatrix_x2(uint32_t r[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(smem_u32(p)));
}

// Position in the ring of shared-memory slots: slot index and the parity of the slot's current round.
struct RingPos {
  int slot;
  uint32_t round;  // number of times the ring has wrapped
  ENG_DEVICE void next(int n) {
    if (++slot == n) {
      slot = 0;
      ++round;
    }
  }
};

// One bounded wait: false once the step has been given up (by this or another CTA).  The clock is read only
// after the first 64 polls, so a wait that is satisfied at once costs nothing.
struct DsWait {
  uint64_t t0;
  uint32_t epoch;
  int n;
  int site;  // DsWaitSite of this wait, recorded if it gives up
};
ENG_DEVICE DsWait ds_wait(uint32_t epoch, int site) { return DsWait{0ull, epoch, 0, site}; }
__device__ int g_ds_layer[1024];  // the layer each CTA is in (diagnostics of a wait that gave up)
__device__ int g_ds_phase[1024];
__device__ int* g_ds_blockdiag;
__device__ __noinline__ bool ds_keep_waiting(const DecodeStepParams& p, DsWait& w) {
  if ((++w.n & 63) != 0) return true;
  if (ld_relaxed_u32(p.epoch + 1) == w.epoch) return false;
  const uint64_t now = global_ns();
  if (w.t0 == 0) {
    w.t0 = now;
  } else if (now - w.t0 > kDsTimeoutNs) {
    atomicExch(p.epoch + 1, w.epoch);
    set_status(p.status, ST_TIMEOUT);
    if (p.diag && atomicCAS(p.diag, 0, w.site) == 0) {
      p.diag[1] = blockIdx.x;
      p.diag[2] = threadIdx.x;
      p.diag[3] = blockIdx.x < 1024 ? g_ds_layer[blockIdx.x] : -1;
    }
    if (g_ds_blockdiag && atomicCAS(g_ds_blockdiag + 4 * blockIdx.x, 0, w.site) == 0) {
      g_ds_blockdiag[4 * blockIdx.x + 1] = threadIdx.x;
      g_ds_blockdiag[4 * blockIdx.x + 2] = blockIdx.x < 1024 ? g_ds_layer[blockIdx.x] : -1;
      g_ds_blockdiag[4 * blockIdx.x + 3] = blockIdx.x < 1024 ? g_ds_phase[blockIdx.x] : -1;
    }
    return false;
  }
  return true;
}

__device__ __noinline__ bool ds_mbar_spin(const DecodeStepParams& p, uint64_t* bar, uint32_t parity, uint32_t epoch,
                                          int site) {
  DsWait w = ds_wait(epoch, site);
  while (!mbar_try(bar, parity)) {
    if (!ds_keep_waiting(p, w)) return false;
    // a full ring means the producer is ahead: it yields the issue slots it shares with a consumer warp
    if (site == WAIT_RING_EMPTY) __nanosleep(200);
  }
  return true;
}
ENG_DEVICE bool ds_mbar_wait(const DecodeStepParams& p, uint64_t* bar, uint32_t parity, uint32_t epoch,
                             int site = WAIT_RING_FULL) {
  return mbar_try(bar, parity) || ds_mbar_spin(p, bar, parity, epoch, site);
}

// Re-polls a word pair (or a single word) until it carries `tag`; the rare, out-of-line part of a wait.
__device__ __noinline__ bool ll_spin2(const DecodeStepParams& p, const unsigned long long* src, unsigned long long* a,
                                      uint32_t tag, uint32_t epoch) {
  DsWait w = ds_wait(epoch, WAIT_STAGE);
  while (ll_tag(a[0]) != tag || ll_tag(a[1]) != tag) {
    if (!ds_keep_waiting(p, w)) return false;
    ll_load2(src, a[0], a[1]);
  }
  return true;
}
__device__ __noinline__ bool ll_spin1(const DecodeStepParams& p, const unsigned long long* src, unsigned long long* a,
                                      uint32_t tag, uint32_t epoch) {
  DsWait w = ds_wait(epoch, WAIT_RESIDUAL);
  while (ll_tag(*a) != tag) {
    if (!ds_keep_waiting(p, w)) return false;
    *a = ll_load1(src);
  }
  return true;
}

// ------------------------------------------------------------------ shared memory

// Keys of one ring chunk of attention: 32 KB of K and V blocks of one KV head.
__host__ __device__ constexpr int ds_blocks_per_chunk(int d) { return kDsSlotBytes / (2 * 16 * d * 2); }

static_assert(sizeof(DsLayer) % 8 == 0, "the layer table is copied in 8-byte words");

struct DsLayout {
  size_t ring, stage, region, red, ts, layers, sched, total;
};
__host__ __device__ inline DsLayout ds_layout(int slots_n, int trows, int kx, int d, int L) {
  const int kpc = 16 * ds_blocks_per_chunk(d);
  DsLayout m;
  m.ring = 0;  // 1024-byte aligned at run time (the layout reserves the slack at the end)
  m.stage = (size_t)slots_n * kDsSlotBytes;
  const size_t stage = (size_t)2 * trows * kx * 2;
  const size_t attn = (size_t)16 * (d + 8) * 2 + (size_t)16 * (kpc + 8) * 2 + (size_t)10 * d * 4 + (size_t)8 * kpc * 4 +
                      (size_t)d * 4 + (size_t)2 * d * 2 + 64;
  m.region = ((stage > attn ? stage : attn) + 127) & ~(size_t)127;
  m.red = m.stage + m.region;
  m.ts = m.red + 8192;
  m.layers = m.ts + 16 * kTsStride * 4;
  m.sched = m.layers + (((size_t)L * sizeof(DsLayer) + 15) & ~(size_t)15);
  m.total = m.sched + (size_t)(DS_PHASES + 1 + kDsMaxItems) * 4 + 1024 + 128;
  return m;
}

size_t decode_step_smem(int slots_n, int trows, int kx, int d, int L) { return ds_layout(slots_n, trows, kx, d, L).total; }

struct DsSmem {
  uint8_t* ring;
  bf16* xs;      // staged activation planes [trows][kx]
  bf16* xl;
  float4* red;   // [8 warps][32 lanes] partial tiles
  float* part;   // [8 tokens][256] per-thread partial sums of squares (aliases red)
  float* ts;     // [16][kTsStride] result tile
  // attention overlay of the staging region
  bf16* qt;      // [16][d + 8]: rows h = hi(q_h), 8 + h = lo(q_h)
  bf16* pt;      // [16][kpc + 8]: probabilities, hi and lo rows
  float* abuf;   // [(G + 2) d]: q heads, k, v of the token
  float* sc;     // [8][kpc] scores
  float* cs;     // [d] cos/sin pairs of the token's position
  bf16* kn;      // [d] new key (bf16, roped)
  bf16* vn;      // [d] new value
  const DsLayer* layers;  // [L] weight pointers
  const int* off;         // [DS_PHASES + 1] this CTA's item ranges
  const int* items;       // this CTA's items
  const int* seq;         // [8] the rows' sequence lengths and positions
  const int* pos;
  uint64_t* full;
  uint64_t* empty;
  float* rstd;   // [8]
  int* ids;      // [8]
  float* mrun;   // [8] online softmax state per head
  float* lrun;
  float* alpha;
  int* flag;
};

// ------------------------------------------------------------------ producer: weights and K/V into the ring

struct DsChunk {
  const void* src[8];  // up to 8 copies (one weight range, or K and V blocks)
  uint32_t dst[8];     // offsets in the slot
  uint32_t bytes[8];
  int n;
};

// Attention item geometry shared by producer and consumer.
struct DsAttnItem {
  int r, g, s, sl, nblk, nsplit, b0, b1;
  bool active;
};
ENG_DEVICE DsAttnItem ds_attn_item(const DecodeStepParams& p, const DsSmem& S, int item) {
  DsAttnItem a;
  a.s = item % p.asplits;
  const int rg = item / p.asplits;
  a.g = rg % p.Hkv;
  a.r = rg / p.Hkv;
  a.sl = S.seq[a.r];
  a.nblk = (a.sl + 15) >> 4;
  if (a.nblk > p.mbs) a.nblk = p.mbs;
  if (a.nblk < 0) a.nblk = 0;
  a.nsplit = (a.nblk + p.ablk - 1) / p.ablk;
  if (a.nsplit < 1) a.nsplit = 1;
  a.active = a.s < a.nsplit;
  a.b0 = a.s * p.ablk;
  a.b1 = min(a.nblk, a.b0 + p.ablk);
  if (a.sl <= 0) a.b1 = a.b0;  // a padding row reads no keys
  return a;
}

ENG_DEVICE int ds_attn_chunks(const DecodeStepParams& p, const DsAttnItem& a) {
  if (!a.active || a.b1 <= a.b0) return 0;
  const int bpc = ds_blocks_per_chunk(p.d);
  return (a.b1 - a.b0 + bpc - 1) / bpc;
}

ENG_DEVICE const bf16* ds_plane(const DecodeStepParams& p, int l, int kv) {
  return p.kv + ((size_t)l * 2 + kv) * (size_t)(p.NB + 1) * p.Hkv * 16 * p.d;
}

// Byte offset of 16-byte chunk cc (8 head-dim values) of key k inside the K (or V) half of a ring chunk:
// each 16-key block holds head_dim / 64 boxes of 16 rows x 128 bytes, rows swizzled in 128-byte units.
ENG_DEVICE uint32_t kv_off(int k, int cc, uint32_t blk_bytes) {
  const int r = k & 15;
  return (uint32_t)(k >> 4) * blk_bytes + (uint32_t)(cc >> 3) * 2048u + (uint32_t)r * 128u +
         (uint32_t)(((cc & 7) ^ (r & 7)) << 4);
}

ENG_DEVICE void ds_producer(const DecodeStepParams& p, const DsSmem& S, uint32_t epoch, uint32_t* issued_out) {
  const int* off = S.off;
  const int NS = p.slots_n;
  uint32_t q = 0;
  RingPos rp{0, 0};
  const int bpc = ds_blocks_per_chunk(p.d);
  const uint32_t blk_bytes = 16u * p.d * 2u;
  for (int l = 0; l < p.L; ++l) {
    const DsLayer& Lw = S.layers[l];
    for (int ph = 0; ph < DS_PHASES; ++ph) {
      for (int it = off[ph]; it < off[ph + 1]; ++it) {
        const int item = S.items[it];
        int nch;
        DsAttnItem a;
        const bf16* W = nullptr;
        int KT = 0;
        if (ph == DS_ATTN) {
          a = ds_attn_item(p, S, item);
          nch = ds_attn_chunks(p, a);
        } else {
          const int K = ph == DS_O ? p.Hq * p.d : ph == DS_DOWN ? p.I : p.H;
          W = ph == DS_QKV ? Lw.qkv : ph == DS_O ? Lw.o : ph == DS_GU ? Lw.gu : Lw.down;
          KT = K >> 5;
          nch = (KT + 31) >> 5;
        }
        for (int c = 0; c < nch; ++c, ++q, rp.next(NS)) {
          const int slot = rp.slot;
          if (rp.round > 0 && !ds_mbar_wait(p, &S.empty[slot], (rp.round - 1) & 1, epoch, WAIT_RING_EMPTY)) {
            *issued_out = q;
            return;
          }
          uint8_t* dst = S.ring + (size_t)slot * kDsSlotBytes;
          if (ph == DS_ATTN) {
            const int bb = a.b0 + c * bpc, be = min(a.b1, bb + bpc);
            mbar_expect_tx(&S.full[slot], (uint32_t)(be - bb) * 2u * blk_bytes);
            for (int b = bb; b < be; ++b) {
              int blk = p.bt[(size_t)a.r * p.mbs + b];
              if (blk < 0 || blk >= p.NB) blk = p.NB;  // flagged by the consumer; the scratch block is harmless
              for (int kv = 0; kv < 2; ++kv) {
                const int row0 = (int)(((((size_t)l * 2 + kv) * (p.NB + 1) + blk) * p.Hkv + a.g) * 16);
                uint8_t* bd = dst + (size_t)kv * bpc * blk_bytes + (size_t)(b - bb) * blk_bytes;
                for (int h = 0; h < p.d / 64; ++h) tma_tile_2d(bd + h * 2048, &p.kv_map, h * 64, row0, &S.full[slot]);
              }
            }
          } else {
            const int nkt = min(32, KT - 32 * c);
            mbar_expect_tx(&S.full[slot], (uint32_t)nkt * 1024u);
            tma_load_1d(dst, W + ((size_t)item * KT + 32 * c) * 512, (uint32_t)nkt * 1024u, &S.full[slot]);
          }
        }
      }
    }
  }
  *issued_out = q;
}

// ------------------------------------------------------------------ consumer pieces

// How a phase's input rows are staged.
enum DsStageMode { STAGE_PLAIN = 0, STAGE_NORM = 1, STAGE_EMBED_NORM = 2, STAGE_FINAL = 3 };

// Stages the T rows of width K of a tagged vector (STAGE_EMBED_NORM: the embedding rows of the step's ids)
// as the hi/lo planes of x * w (STAGE_PLAIN: x itself), with each row's 1 / rms(x) for the norm modes.
// STAGE_FINAL writes the LM head's inputs instead: the rows themselves, the planes of x * w in global
// memory and each row's sum of squares.  Up to 8 word pairs per thread are in flight at once; one copy of
// this code serves every phase.
ENG_DEVICE bool ds_stage(const DecodeStepParams& p, const DsSmem& S, const unsigned long long* src, uint32_t tag,
                         int K, const float* w, int mode, uint32_t epoch) {
  const int tid = threadIdx.x;
  const bool norm = mode != STAGE_PLAIN;
  if (norm)
    for (int t = 0; t < p.T; ++t) S.part[t * kDsConsumers + tid] = 0.f;
  int cur = -1;
  float run = 0.f;
  bool ok = true;
  const int npairs = p.T * K / 2;
  for (int base = tid; base < npairs && ok; base += kDsConsumers * 8) {
    unsigned long long a[8][2];
    float2 wv[8];
    float sq[8];           // each pair's sum of squares, added in pair order below (a fixed summation order)
    unsigned pending = 0;  // pairs of this round not yet seen with the tag
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int pi = base + j * kDsConsumers;
      if (pi < npairs) {
        const int i = 2 * pi, t = i / K, c = i - t * K;
        if (mode == STAGE_EMBED_NORM) {
          const int id = S.ids[t];
          a[j][0] = ((unsigned long long)tag << 32) | __float_as_uint(__bfloat162float(p.embed[packed_offset(id, c, K)]));
          a[j][1] = ((unsigned long long)tag << 32) | __float_as_uint(__bfloat162float(p.embed[packed_offset(id, c + 1, K)]));
        } else {
          ll_load2(src + i, a[j][0], a[j][1]);
        }
        wv[j] = norm ? make_float2(__ldg(w + c), __ldg(w + c + 1)) : make_float2(1.f, 1.f);
        pending |= 1u << j;
      }
    }
    // take every pair whose words carry the tag; re-poll the rest together, one round trip per round
    DsWait wt = ds_wait(epoch, WAIT_STAGE);
    while (true) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (!(pending & (1u << j)) || ll_tag(a[j][0]) != tag || ll_tag(a[j][1]) != tag) continue;
        pending &= ~(1u << j);
        const int i = 2 * (base + j * kDsConsumers), t = i / K, c = i - t * K;
        const float v0 = ll_val(a[j][0]), v1 = ll_val(a[j][1]);
        sq[j] = v0 * v0 + v1 * v1;
        if (mode == STAGE_FINAL) {
          p.h_out[i] = v0;
          p.h_out[i + 1] = v1;
          put_split2(p.xn_h, p.xn_l, (size_t)i, v0 * wv[j].x, v1 * wv[j].y);
        } else {
          uint32_t h, lo;
          split_bf16x2(v0 * wv[j].x, v1 * wv[j].y, h, lo);
          *reinterpret_cast<uint32_t*>(S.xs + (size_t)t * p.kx + c) = h;
          *reinterpret_cast<uint32_t*>(S.xl + (size_t)t * p.kx + c) = lo;
        }
      }
      if (!pending) break;
      if (!ds_keep_waiting(p, wt)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (pending & (1u << j)) ll_load2(src + 2 * (base + j * kDsConsumers), a[j][0], a[j][1]);
    }
    if (norm && ok) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int pi = base + j * kDsConsumers;
        if (pi >= npairs) break;
        const int t = (2 * pi) / K;
        if (t != cur) {
          if (cur >= 0) S.part[cur * kDsConsumers + tid] = run;
          cur = t;
          run = 0.f;
        }
        run += sq[j];
      }
    }
  }
  if (norm && cur >= 0) S.part[cur * kDsConsumers + tid] = run;
  if (!csync_and(ok)) return false;
  if (norm) {
    const int warp = tid >> 5, lane = tid & 31;
    for (int tw = warp; tw < p.T; tw += kDsWarps) {
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < kDsWarps; ++j) ss += S.part[tw * kDsConsumers + lane + 32 * j];
      ss = warp_sum(ss);
      if (lane == 0) {
        if (mode == STAGE_FINAL)
          p.sq[(size_t)tw * p.sq_stride] = ss;
        else
          S.rstd[tw] = rsqrtf(ss / (float)K + p.eps);
      }
    }
    csync();
  }
  return true;
}

// Attention splits of a row of length sl.  A padding row (length 0) has one, which publishes a zero output:
// the output projection's staging then waits for every row's attention items, which keeps each reader of
// the QKV words upstream of their next writer.
ENG_DEVICE int ds_row_splits(const DecodeStepParams& p, int sl) {
  if (sl <= 0) return 1;
  const int nblk = min((sl + 15) >> 4, p.mbs);
  return max(1, (nblk + p.ablk - 1) / p.ablk);
}

// The output projection's input: each row's attention output merged from its splits' (O, max, sum) words
// in split order -- M = the largest max, w_s = 2^(max_s - M), out = (sum_s w_s O_s) / (sum_s w_s sum_s) -- and
// staged as hi/lo planes (a padding row's single split publishes zeros).  Every split's words of a round
// are requested together.
ENG_DEVICE bool ds_stage_attn(const DecodeStepParams& p, const DsSmem& S, uint32_t tag, uint32_t epoch) {
  const int tid = threadIdx.x, d = p.d, G = p.Hq / p.Hkv, Hq = p.Hq, SP = p.asplits;
  const size_t wrow = (size_t)(d + 2);
  float* wt = S.part;  // [T][Hq][kDsMaxSplits]: each split's weight with 1 / (sum of weighted sums) folded in
  bool ok = true;
  for (int idx = tid; idx < p.T * Hq && ok; idx += kDsConsumers) {
    const int t = idx / Hq, h = idx - t * Hq;
    const int ns = ds_row_splits(p, S.seq[t]);
    const unsigned long long* base =
        p.attn_ws + (((size_t)t * p.Hkv + h / G) * SP) * G * wrow + (size_t)(h % G) * wrow + d;
    unsigned long long w2[kDsMaxSplits][2];
#pragma unroll
    for (int sp = 0; sp < kDsMaxSplits; ++sp)
      if (sp < ns) ll_load2(base + (size_t)sp * G * wrow, w2[sp][0], w2[sp][1]);
    DsWait wt_ = ds_wait(epoch, WAIT_ATTN_STATS);
    while (true) {
      bool all = true;
#pragma unroll
      for (int sp = 0; sp < kDsMaxSplits; ++sp)
        all = all && (sp >= ns || (ll_tag(w2[sp][0]) == tag && ll_tag(w2[sp][1]) == tag));
      if (all) break;
      if (!ds_keep_waiting(p, wt_)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int sp = 0; sp < kDsMaxSplits; ++sp)
        if (sp < ns && (ll_tag(w2[sp][0]) != tag || ll_tag(w2[sp][1]) != tag))
          ll_load2(base + (size_t)sp * G * wrow, w2[sp][0], w2[sp][1]);
    }
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < kDsMaxSplits; ++sp)
      if (sp < ns) M = fmaxf(M, ll_val(w2[sp][0]));
    float L = 0.f, wv[kDsMaxSplits];
#pragma unroll
    for (int sp = 0; sp < kDsMaxSplits; ++sp) {
      wv[sp] = sp < ns ? exp2f(ll_val(w2[sp][0]) - M) : 0.f;
      L += sp < ns ? ll_val(w2[sp][1]) * wv[sp] : 0.f;
    }
#pragma unroll
    for (int sp = 0; sp < kDsMaxSplits; ++sp) wt[idx * kDsMaxSplits + sp] = ns ? wv[sp] / L : 0.f;
  }
  if (!csync_and(ok)) return false;
  const int width = Hq * d, npairs = p.T * width / 2;
  for (int base = tid; base < npairs && ok; base += kDsConsumers * 4) {
    unsigned long long a[4][kDsMaxSplits][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int pi = base + j * kDsConsumers;
      if (pi >= npairs) continue;
      const int i = 2 * pi, t = i / width, h = (i - t * width) / d, col = i - t * width - h * d;
      const int ns = ds_row_splits(p, S.seq[t]);
      const unsigned long long* at =
          p.attn_ws + (((size_t)t * p.Hkv + h / G) * SP) * G * wrow + (size_t)(h % G) * wrow + col;
#pragma unroll
      for (int sp = 0; sp < kDsMaxSplits; ++sp)
        if (sp < ns) ll_load2(at + (size_t)sp * G * wrow, a[j][sp][0], a[j][sp][1]);
    }
    DsWait wt_ = ds_wait(epoch, WAIT_ATTN_OUT);
    while (true) {
      bool all = true;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pi = base + j * kDsConsumers;
        if (pi >= npairs) continue;
        const int ns = ds_row_splits(p, S.seq[(2 * pi) / width]);
#pragma unroll
        for (int sp = 0; sp < kDsMaxSplits; ++sp)
          all = all && (sp >= ns || (ll_tag(a[j][sp][0]) == tag && ll_tag(a[j][sp][1]) == tag));
      }
      if (all) break;
      if (!ds_keep_waiting(p, wt_)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pi = base + j * kDsConsumers;
        if (pi >= npairs) continue;
        const int i = 2 * pi, t = i / width, h = (i - t * width) / d, col = i - t * width - h * d;
        const int ns = ds_row_splits(p, S.seq[t]);
        const unsigned long long* at =
            p.attn_ws + (((size_t)t * p.Hkv + h / G) * SP) * G * wrow + (size_t)(h % G) * wrow + col;
#pragma unroll
        for (int sp = 0; sp < kDsMaxSplits; ++sp)
          if (sp < ns && (ll_tag(a[j][sp][0]) != tag || ll_tag(a[j][sp][1]) != tag))
            ll_load2(at + (size_t)sp * G * wrow, a[j][sp][0], a[j][sp][1]);
      }
    }
    if (!ok) break;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int pi = base + j * kDsConsumers;
      if (pi >= npairs) continue;
      const int i = 2 * pi, t = i / width, h = (i - t * width) / d, col = i - t * width - h * d;
      const int ns = ds_row_splits(p, S.seq[t]);
      float o0 = 0.f, o1 = 0.f;
#pragma unroll
      for (int sp = 0; sp < kDsMaxSplits; ++sp)
        if (sp < ns) {
          const float wgt = wt[(t * Hq + h) * kDsMaxSplits + sp];
          o0 += ll_val(a[j][sp][0]) * wgt;
          o1 += ll_val(a[j][sp][1]) * wgt;
        }
      uint32_t hi, lo;
      split_bf16x2(o0, o1, hi, lo);
      *reinterpret_cast<uint32_t*>(S.xs + (size_t)t * p.kx + h * d + col) = hi;
      *reinterpret_cast<uint32_t*>(S.xl + (size_t)t * p.kx + h * d + col) = lo;
    }
  }
  return csync_and(ok);
}

// This token's q heads, k and v of one KV head from the QKV phase's words into S.abuf [(G + 2) d] (fp32).
ENG_DEVICE bool ds_gather_head(const DecodeStepParams& p, const DsSmem& S, const unsigned long long* qrow, int g,
                               uint32_t tag, uint32_t epoch) {
  const int d = p.d, G = p.Hq / p.Hkv;
  const int gq = g * G * d, gk = (p.Hq + g) * d, gv = (p.Hq + p.Hkv + g) * d;
  const int npairs = (G + 2) * d / 2;
  for (int base = threadIdx.x; base < npairs; base += kDsConsumers * 4) {
    unsigned long long a[4][2];
    const unsigned long long* at[4];
    unsigned pending = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int pi = base + j * kDsConsumers, i = 2 * pi;
      at[j] = qrow + (i < G * d ? gq + i : i < (G + 1) * d ? gk + i - G * d : gv + i - (G + 1) * d);
      if (pi < npairs) {
        ll_load2(at[j], a[j][0], a[j][1]);
        pending |= 1u << j;
      }
    }
    DsWait wt = ds_wait(epoch, WAIT_HEAD);
    while (true) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!(pending & (1u << j)) || ll_tag(a[j][0]) != tag || ll_tag(a[j][1]) != tag) continue;
        pending &= ~(1u << j);
        const int pi = base + j * kDsConsumers;
        S.abuf[2 * pi] = ll_val(a[j][0]);
        S.abuf[2 * pi + 1] = ll_val(a[j][1]);
      }
      if (!pending) break;
      if (!ds_keep_waiting(p, wt)) return false;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (pending & (1u << j)) ll_load2(at[j], a[j][0], a[j][1]);
    }
  }
  return true;
}

// One 16-row tile of a packed weight ([N][K]) against the staged planes: the tile's chunks from the ring,
// every warp taking every 8th k-tile into four independent accumulator chains (two k-steps x hi/lo planes),
// then the warps summed in order.  Returns, in the first 32 threads, the tile's values in MMA fragment
// order: v = (row r, token c), (r, c + 1), (r + 8, c), (r + 8, c + 1) with r = tid / 4, c = 2 (tid % 4).
// The activation fragment comes from 32-bit shared loads (a row past the step's tokens reads row 0, so
// lanes of one step's rows read the same words as a broadcast).
ENG_DEVICE bool ds_gemv(const DecodeStepParams& p, const DsSmem& S, int K, RingPos& rp, uint32_t epoch, float4& v) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KT = K >> 5;
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
  float c2[4] = {0.f, 0.f, 0.f, 0.f}, c3[4] = {0.f, 0.f, 0.f, 0.f};
  const int g = lane >> 2;
  const int xrow = g < p.T ? g : 0;
  const uint32_t* xs = reinterpret_cast<const uint32_t*>(S.xs + (size_t)xrow * p.kx) + (lane & 3);
  const uint32_t* xl = reinterpret_cast<const uint32_t*>(S.xl + (size_t)xrow * p.kx) + (lane & 3);
  bool ok = true;
  for (int c = 0; c * 32 < KT; ++c, rp.next(p.slots_n)) {
    if (!ds_mbar_wait(p, &S.full[rp.slot], rp.round & 1, epoch)) {
      ok = false;
      break;
    }
    const uint4* w = reinterpret_cast<const uint4*>(S.ring + (size_t)rp.slot * kDsSlotBytes) + lane;
    const int nkt = min(32, KT - 32 * c);
    const uint32_t* xsc = xs + 32 * c * 16;
    const uint32_t* xlc = xl + 32 * c * 16;
#pragma unroll 4
    for (int kt = warp; kt < nkt; kt += kDsWarps) {
      const uint4 a0 = w[kt * 64], a1 = w[kt * 64 + 32];
      const uint32_t* xh = xsc + kt * 16;
      const uint32_t* xo = xlc + kt * 16;
      mma_bf16(c0, a0.x, a0.y, a0.z, a0.w, xh[0], xh[4]);
      mma_bf16(c1, a1.x, a1.y, a1.z, a1.w, xh[8], xh[12]);
      mma_bf16(c2, a0.x, a0.y, a0.z, a0.w, xo[0], xo[4]);
      mma_bf16(c3, a1.x, a1.y, a1.z, a1.w, xo[8], xo[12]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[rp.slot]);
  }
  if (ok)
    S.red[warp * 32 + lane] = make_float4((c0[0] + c1[0]) + (c2[0] + c3[0]), (c0[1] + c1[1]) + (c2[1] + c3[1]),
                                          (c0[2] + c1[2]) + (c2[2] + c3[2]), (c0[3] + c1[3]) + (c2[3] + c3[3]));
  if (!csync_and(ok)) return false;
  if (tid < 32) {
    v = S.red[tid];
    for (int w2 = 1; w2 < kDsWarps; ++w2) {
      const float4 u = S.red[w2 * 32 + tid];
      v.x += u.x;
      v.y += u.y;
      v.z += u.z;
      v.w += u.w;
    }
  }
  return true;
}

// Attention of one item: request row r, KV head g, key split s.  QK-norm and RoPE of the token's q heads
// and k, the write of the new K/V (by the split holding the new position), online softmax over the item's
// chunks, and the merge of the row's splits by the split that finishes last, in split order.
ENG_DEVICE bool ds_attention(const DecodeStepParams& p, const DsSmem& S, int l, int item, RingPos& rp, uint32_t& q,
                             uint32_t tag_in, uint32_t tag_out, uint32_t epoch) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = p.d, G = p.Hq / p.Hkv, E = d / 32;
  const int bpc = ds_blocks_per_chunk(d), kpc = 16 * bpc;
  const DsAttnItem a = ds_attn_item(p, S, item);
  if (!a.active) return true;
  const int t = a.r;  // decode-only step: token t is request row t
  const int QKV = (p.Hq + 2 * p.Hkv) * d;
  const unsigned long long* qrow = p.qkv_ll + (size_t)t * QKV;
  int pos = S.pos[t];
  const bool pos_ok = pos >= 0 && pos < p.max_pos && (pos >> 4) < p.mbs;
  if (!pos_ok) pos = 0;
  if (tid == 0 && a.s == 0 && a.g == 0 && a.sl > 0 && (!pos_ok || ((a.sl + 15) >> 4) > p.mbs))
    set_status(p.status, ST_BAD_POSITION);

  // ---- loads that do not depend on this step's projections go first: the RoPE row, the QK-norm weights
  for (int i = tid; i < d; i += kDsConsumers) S.cs[i] = p.rope[(size_t)pos * d + i];
  float nwv[2][4];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int row = warp + kDsWarps * k;
    const float* nw = row < G ? S.layers[l].q_norm : row == G ? S.layers[l].k_norm : nullptr;
#pragma unroll
    for (int e = 0; e < 4; ++e) nwv[k][e] = (nw && e < E) ? __ldg(nw + lane * E + e) : 1.f;
  }
  // ---- this token's q heads, k and v
  bool ok = ds_gather_head(p, S, qrow, a.g, tag_in, epoch);
  for (int i = tid; i < 16 * (d + 8); i += kDsConsumers) S.qt[i] = __float2bfloat16_rn(0.f);
  for (int i = tid; i < 16 * (kpc + 8); i += kDsConsumers) S.pt[i] = __float2bfloat16_rn(0.f);
  if (tid < 8) {
    S.mrun[tid] = -INFINITY;
    S.lrun[tid] = 0.f;
  }
  if (!csync_and(ok)) return false;

  // ---- QK-norm and rotate-half RoPE (warp per head row: q heads, then k); v is only rounded
  const bool qk_norm = S.layers[l].q_norm != nullptr;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int row = warp + kDsWarps * k;
    if (row >= G + 2) break;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) x[e] = S.abuf[row * d + lane * E + e];
    if (row <= G) {
      if (qk_norm) {
        float ss = 0.f;
        _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) ss += x[e] * x[e];
        ss = warp_sum(ss);
        const float rs = rsqrtf(ss / (float)d + p.eps);
        _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) x[e] = x[e] * rs * nwv[k][e];
      }
      float y[4] = {0.f, 0.f, 0.f, 0.f};
      _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) {
        const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
        const int ii = (lane & 15) * E + e;
        const float c = S.cs[2 * ii], sn = S.cs[2 * ii + 1];
        y[e] = (lane < 16) ? (x[e] * c - other * sn) : (x[e] * c + other * sn);
      }
      _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) x[e] = y[e];
    }
    if (row < G) {
      _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) {
        const bf16 h = __float2bfloat16_rn(x[e]);
        S.qt[row * (d + 8) + lane * E + e] = h;
        S.qt[(8 + row) * (d + 8) + lane * E + e] = __float2bfloat16_rn(x[e] - __bfloat162float(h));
      }
    } else {
      bf16* dstv = row == G ? S.kn : S.vn;
      _Pragma("unroll") for (int e = 0; e < 4; ++e) if (e < E) dstv[lane * E + e] = __float2bfloat16_rn(x[e]);
    }
  }
  csync();

  // ---- the new K/V into the paged pool (the split that holds the new position; padding: scratch block)
  if (a.s == a.nsplit - 1) {
    int slot = -1;
    if (a.sl > 0) {
      if (!pos_ok) {
        slot = -2;
      } else {
        const int b = p.bt[(size_t)a.r * p.mbs + (pos >> 4)];
        slot = (b < 0 || b >= p.NB) ? -3 : b * 16 + (pos & 15);
      }
    }
    const int blk = slot >= 0 ? slot >> 4 : p.NB, off = slot >= 0 ? slot & 15 : 0;
    const size_t o = (((size_t)blk * p.Hkv + a.g) * 16 + off) * d;
    bf16* kp = const_cast<bf16*>(ds_plane(p, l, 0)) + o;
    bf16* vp = const_cast<bf16*>(ds_plane(p, l, 1)) + o;
    for (int i = tid; i < d / 2; i += kDsConsumers) {
      reinterpret_cast<uint32_t*>(kp)[i] = reinterpret_cast<const uint32_t*>(S.kn)[i];
      reinterpret_cast<uint32_t*>(vp)[i] = reinterpret_cast<const uint32_t*>(S.vn)[i];
    }
    if (tid == 0 && a.g == 0) {
      p.slots[t] = slot >= 0 ? slot : -1;
      if (slot < -1) set_status(p.status, slot == -2 ? ST_BAD_POSITION : ST_BAD_BLOCK);
    }
  }
  const size_t wrow = (size_t)(d + 2);
  unsigned long long* ws = p.attn_ws + (((size_t)t * p.Hkv + a.g) * p.asplits) * G * wrow;  // [split][G][d + 2]
  if (a.sl <= 0) {  // a padding row attends to nothing: O = 0 with max 0 and sum 1 (a zero output)
    for (int i = tid; i < G * (int)wrow; i += kDsConsumers) {
      const int col = i % (int)wrow;
      ll_store(ws + i, col == d + 1 ? 1.f : 0.f, tag_out);
    }
    return true;
  }

  // ---- online softmax over the item's chunks (base 2)
  const int gl = lane >> 2, tl = lane & 3;  // MMA fragment row group and column pair of this lane
  const int nd = d / 8;                     // 8-column tiles of the output
  constexpr int kOt = (16 + kDsWarps - 1) / kDsWarps;  // output column tiles per warp (d / 8 <= 16)
  float o[kOt][4];
#pragma unroll
  for (int j = 0; j < kOt; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  const int nch = ds_attn_chunks(p, a);
  const uint32_t blk_bytes = 16u * d * 2u;
  for (int c = 0; c < nch; ++c, rp.next(p.slots_n), ++q) {
    const int slot = rp.slot;
    if (!ds_mbar_wait(p, &S.full[slot], rp.round & 1, epoch)) ok = false;
    if (!csync_and(ok)) return false;
    bf16* Kc = reinterpret_cast<bf16*>(S.ring + (size_t)slot * kDsSlotBytes);
    bf16* Vc = reinterpret_cast<bf16*>(S.ring + (size_t)slot * kDsSlotBytes + (size_t)bpc * blk_bytes);
    const int bb = a.b0 + c * bpc, nb = min(a.b1, bb + bpc) - bb;
    const int key0 = bb * 16, kb = nb * 16;
    // the new position's key and value (the pool copy may predate this step), and zero values for keys
    // past the row's length (a freed block's stale contents must not reach the product)
    uint8_t* Kb = reinterpret_cast<uint8_t*>(Kc);
    uint8_t* Vb = reinterpret_cast<uint8_t*>(Vc);
    if (pos >= key0 && pos < key0 + kb && tid < d / 4) {  // one 16-byte chunk of K or V per thread
      const int cc = tid % (d / 8);
      uint8_t* dstc = (tid < d / 8 ? Kb : Vb) + kv_off(pos - key0, cc, blk_bytes);
      *reinterpret_cast<uint4*>(dstc) = reinterpret_cast<const uint4*>(tid < d / 8 ? S.kn : S.vn)[cc];
    }
    const int kvalid = min(kb, a.sl - key0);
    for (int i = tid; i < (kb - kvalid) * (d / 8); i += kDsConsumers)
      *reinterpret_cast<uint4*>(Vb + kv_off(kvalid + i / (d / 8), i % (d / 8), blk_bytes)) = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes before the slot's next copy
    csync();

    // S = Q K^T: warp w takes the 8-key tiles w, w + 8
    for (int nt = warp; nt < kb / 8; nt += kDsWarps) {
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int ks = 0; ks < d / 16; ks += 2) {
        uint32_t af[4], af2[4], bfr[4];
        ldmatrix_x4(af, S.qt + (size_t)(lane & 15) * (d + 8) + ks * 16 + (lane >> 4) * 8);
        ldmatrix_x4(af2, S.qt + (size_t)(lane & 15) * (d + 8) + (ks + 1) * 16 + (lane >> 4) * 8);
        ldmatrix_x4(bfr, Kb + kv_off(nt * 8 + (lane & 7), 2 * ks + (lane >> 3), blk_bytes));
        mma_bf16(sacc, af[0], af[1], af[2], af[3], bfr[0], bfr[1]);
        mma_bf16(sacc, af2[0], af2[1], af2[2], af2[3], bfr[2], bfr[3]);
      }
      if (gl < G) {
        const int k = nt * 8 + 2 * tl;
        const float s0 = (sacc[0] + sacc[2]) * p.scale_log2, s1 = (sacc[1] + sacc[3]) * p.scale_log2;
        S.sc[gl * kpc + k] = key0 + k < a.sl ? s0 : -INFINITY;
        S.sc[gl * kpc + k + 1] = key0 + k + 1 < a.sl ? s1 : -INFINITY;
      }
    }
    csync();
    // per head (a warp each): the chunk's maximum, the probabilities as hi/lo rows, the running sum
    for (int hh = warp; hh < G; hh += kDsWarps) {
      float mx = -INFINITY;
      for (int k = lane; k < kb; k += 32) mx = fmaxf(mx, S.sc[hh * kpc + k]);
      mx = warp_max(mx);
      const float m_old = S.mrun[hh], m_new = fmaxf(m_old, mx);
      float sum = 0.f;
      for (int k = lane; k < kb; k += 32) {
        const float pr = exp2f(S.sc[hh * kpc + k] - m_new);
        const bf16 h = __float2bfloat16_rn(pr);
        S.pt[hh * (kpc + 8) + k] = h;
        S.pt[(8 + hh) * (kpc + 8) + k] = __float2bfloat16_rn(pr - __bfloat162float(h));
        sum += pr;
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        const float al = exp2f(m_old - m_new);
        S.alpha[hh] = al;
        S.lrun[hh] = S.lrun[hh] * al + sum;
        S.mrun[hh] = m_new;
      }
    }
    csync();
    // O = alpha O + P V: warp w owns the output column tiles w, w + 7, w + 14
    const float al = gl < G ? S.alpha[gl] : 1.f;
#pragma unroll
    for (int j = 0; j < kOt; ++j) {
      const int ndt = warp + kDsWarps * j;
      if (ndt >= nd) continue;
      o[j][0] *= al;
      o[j][1] *= al;
      o[j][2] *= al;
      o[j][3] *= al;
      for (int ks = 0; ks < kb / 16; ++ks) {
        uint32_t af[4], bfr[2];
        ldmatrix_x4(af, S.pt + (size_t)(lane & 15) * (kpc + 8) + ks * 16 + (lane >> 4) * 8);
        uint32_t tr[4];
        ldmatrix_x4_trans(tr, Vb + kv_off(ks * 16 + (lane & 15), ndt, blk_bytes));
        bfr[0] = tr[0];
        bfr[1] = tr[1];
        mma_bf16(o[j], af[0], af[1], af[2], af[3], bfr[0], bfr[1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
    csync();  // the score and probability tiles are rewritten by the next chunk
  }

  // ---- this split's (O unnormalised, running max, running sum) as tagged words; the output projection's
  // staging merges a row's splits in split order
  if (gl < G) {
#pragma unroll
    for (int j = 0; j < kOt; ++j) {
      const int ndt = warp + kDsWarps * j;
      if (ndt >= nd) continue;
      unsigned long long* dst = ws + ((size_t)a.s * G + gl) * wrow + ndt * 8 + 2 * tl;
      ll_store(dst, o[j][0] + o[j][2], tag_out);
      ll_store(dst + 1, o[j][1] + o[j][3], tag_out);
    }
  }
  if (tid < G) {
    ll_store(ws + ((size_t)a.s * G + tid) * wrow + d, S.mrun[tid], tag_out);
    ll_store(ws + ((size_t)a.s * G + tid) * wrow + d + 1, S.lrun[tid], tag_out);
  }
  return true;
}

ENG_DEVICE uint32_t ds_tag(uint32_t epoch, int l, int ph) { return (epoch << 8) | (uint32_t)(l * DS_PHASES + ph + 1); }

// Epilogue of one tile of a projection phase, in the first 32 threads, each holding four values of the tile
// (rows r, r + 8 and tokens c, c + 1 with r = tid / 4, c = 2 (tid % 4); ds_gemv):
//   QKV   the raw projection (+ bias), 1 / rms of the input applied, for the attention items;
//   O     h = h_prev (the previous layer's output, or the embedding in layer 0) + the tile;
//   GU    silu(gate) * up: tile rows 0..7 are gate rows and rows 8..15 the matching up rows;
//   DOWN  h = h after O + the tile.
// pre[k]: the residual words of (row r + 8 (k / 2), token c + k % 2), requested before the product.
ENG_DEVICE bool ds_epilogue(const DecodeStepParams& p, const DsSmem& S, int ph, int tile, const DsLayer& Lw,
                            const unsigned long long* hres, const unsigned long long (&pre)[4], uint32_t tres,
                            uint32_t tout, uint32_t epoch, const float4& v) {
  const int tid = threadIdx.x;
  if (tid >= 32) return true;
  const int r = tid >> 2, c = 2 * (tid & 3);
  const float val[4] = {v.x, v.y, v.z, v.w};
  if (ph == DS_GU) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = c + k;
      if (t >= p.T) continue;
      const float ga = val[k] * S.rstd[t], up = val[2 + k] * S.rstd[t];
      ll_store(p.act_ll + (size_t)t * p.I + tile * 8 + r, ga / (1.f + expf(-ga)) * up, tout);
    }
    return true;
  }
  const int QKV = (p.Hq + 2 * p.Hkv) * p.d;
  bool ok = true;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int t = c + (k & 1), row = tile * 16 + r + 8 * (k >> 1);
    if (t >= p.T) continue;
    if (ph == DS_QKV) {
      ll_store(p.qkv_ll + (size_t)t * QKV + row, val[k] * S.rstd[t] + (Lw.qkv_bias ? Lw.qkv_bias[row] : 0.f), tout);
      continue;
    }
    float old;
    if (hres) {
      unsigned long long wd = pre[k];
      if (ll_tag(wd) != tres && !ll_spin1(p, hres + (size_t)t * p.H + row, &wd, tres, epoch)) {
        ok = false;
        continue;
      }
      old = ll_val(wd);
    } else {
      old = __bfloat162float(p.embed[packed_offset(S.ids[t], row, p.H)]);
    }
    ll_store(p.h_ll + (size_t)t * p.H + row, old + val[k], tout);
  }
  return ok;
}

ENG_DEVICE void ds_consumer(const DecodeStepParams& p, const DsSmem& S, uint32_t epoch, uint32_t* consumed) {
  const int tid = threadIdx.x;
  RingPos rp{0, 0};
  uint32_t q = 0;  // chunks consumed
  bool ok = true;
  for (int l = 0; l < p.L && ok; ++l) {
    const DsLayer& Lw = S.layers[l];
    if (tid == 0 && blockIdx.x < 1024) g_ds_layer[blockIdx.x] = l;
    for (int ph = 0; ph < DS_PHASES && ok; ++ph) {
      const int first = S.off[ph], last = S.off[ph + 1];
      if (first == last) continue;
      if (tid == 0 && blockIdx.x < 1024) g_ds_phase[blockIdx.x] = ph;
      if (ph == DS_ATTN) {
        for (int it = first; ok && it < last; ++it)
          ok = ds_attention(p, S, l, S.items[it], rp, q, ds_tag(epoch, l, DS_QKV), ds_tag(epoch, l, DS_ATTN), epoch);
        continue;
      }
      // the phase's input rows, and for O and DOWN the residual they add to
      const unsigned long long* src = p.h_ll;
      uint32_t tag = ds_tag(epoch, l, DS_O);
      int K = p.H, mode = STAGE_NORM;
      const float* w = Lw.post_norm;
      const unsigned long long* hres = p.h_ll;
      uint32_t tres = ds_tag(epoch, l, DS_O);
      if (ph == DS_QKV) {
        src = l ? p.h_ll : nullptr;
        tag = l ? ds_tag(epoch, l - 1, DS_DOWN) : 0u;
        w = Lw.in_norm;
        mode = l ? STAGE_NORM : STAGE_EMBED_NORM;
      } else if (ph == DS_O) {
        src = nullptr;  // the attention splits' words (ds_stage_attn)
        tag = ds_tag(epoch, l, DS_ATTN);
        K = p.Hq * p.d;
        w = nullptr;
        mode = STAGE_PLAIN;
        hres = l ? p.h_ll : nullptr;
        tres = l ? ds_tag(epoch, l - 1, DS_DOWN) : 0u;
      } else if (ph == DS_DOWN) {
        src = p.act_ll;
        tag = ds_tag(epoch, l, DS_GU);
        K = p.I;
        w = nullptr;
        mode = STAGE_PLAIN;
      }
      const bool resid = ph == DS_O || ph == DS_DOWN;
      ok = ph == DS_O ? ds_stage_attn(p, S, tag, epoch) : ds_stage(p, S, src, tag, K, w, mode, epoch);
      for (int it = first; ok && it < last; ++it) {
        const int tile = S.items[it];
        // the residual words this thread adds to, requested before the product so that they overlap the MMAs
        unsigned long long pre[4] = {0ull, 0ull, 0ull, 0ull};
        if (resid && hres && tid < 32) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int t = 2 * (tid & 3) + (k & 1), row = tile * 16 + (tid >> 2) + 8 * (k >> 1);
            if (t < p.T) pre[k] = ll_load1(hres + (size_t)t * p.H + row);
          }
        }
        const uint32_t nch = (uint32_t)((K / 32 + 31) / 32);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        ok = ds_gemv(p, S, K, rp, epoch, v) &&
             csync_and(ds_epilogue(p, S, ph, tile, Lw, resid ? hres : nullptr, pre, tres, ds_tag(epoch, l, ph), epoch, v));
        q += nch;
      }
    }
    ok = csync_and(ok);
  }
  // ---- the final residual for the LM head: planes of h * final norm weight and each row's sum of squares
  if (ok && blockIdx.x == 0)
    ds_stage(p, S, p.h_ll, ds_tag(epoch, p.L - 1, DS_DOWN), p.H, p.final_norm, STAGE_FINAL, epoch);
  if (tid == 0) *consumed = q;
}

__global__ void __launch_bounds__(kDsThreads, 1) k_decode_step(const __grid_constant__ DecodeStepParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t s_full[kDsMaxSlots], s_empty[kDsMaxSlots];
  __shared__ float s_rstd[8], s_m[8], s_l[8], s_alpha[8];
  __shared__ int s_ids[8], s_flag[1], s_seq[8], s_pos[8];
  __shared__ uint32_t s_issued, s_consumed;
  const DsLayout lay = ds_layout(p.slots_n, p.trows, p.kx, p.d, p.L);
  DsSmem S;
  // every region at a fixed offset from a 1024-byte aligned base (the swizzled tensor copies need it)
  uint8_t* const sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem) + 1023) & ~static_cast<uintptr_t>(1023));
  S.ring = sbase + lay.ring;
  S.xs = reinterpret_cast<bf16*>(sbase + lay.stage);
  S.xl = S.xs + (size_t)p.trows * p.kx;
  S.red = reinterpret_cast<float4*>(sbase + lay.red);
  S.part = reinterpret_cast<float*>(sbase + lay.red);
  S.ts = reinterpret_cast<float*>(sbase + lay.ts);
  {
    const int kpc = 16 * ds_blocks_per_chunk(p.d);
    uint8_t* o = sbase + lay.stage;
    S.qt = reinterpret_cast<bf16*>(o);
    o += (size_t)16 * (p.d + 8) * 2;
    S.pt = reinterpret_cast<bf16*>(o);
    o += (size_t)16 * (kpc + 8) * 2;
    S.abuf = reinterpret_cast<float*>(o);
    o += (size_t)10 * p.d * 4;
    S.sc = reinterpret_cast<float*>(o);
    o += (size_t)8 * kpc * 4;
    S.cs = reinterpret_cast<float*>(o);
    o += (size_t)p.d * 4;
    S.kn = reinterpret_cast<bf16*>(o);
    S.vn = S.kn + p.d;
  }
  S.layers = reinterpret_cast<const DsLayer*>(sbase + lay.layers);
  int* s_sched = reinterpret_cast<int*>(sbase + lay.sched);
  S.off = s_sched;
  S.items = s_sched + DS_PHASES + 1;
  S.seq = s_seq;
  S.pos = s_pos;
  S.full = s_full;
  S.empty = s_empty;
  S.rstd = s_rstd;
  S.ids = s_ids;
  S.mrun = s_m;
  S.lrun = s_l;
  S.alpha = s_alpha;
  S.flag = s_flag;
  const uint32_t epoch = ld_relaxed_u32(p.epoch);
  if (threadIdx.x == 0 && blockIdx.x == 0) g_ds_blockdiag = p.diag ? p.diag + 4 : nullptr;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.slots_n; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kDsWarps);
    }
    s_issued = s_consumed = 0;
  }
  {  // this CTA's schedule, the layer table and the rows' lengths and positions, read once per step
    const int* goff = p.sched_off + (size_t)blockIdx.x * (DS_PHASES + 1);
    const int first = goff[0];
    for (int i = threadIdx.x; i <= DS_PHASES; i += blockDim.x) s_sched[i] = goff[i] - first;
    const int n = min(goff[DS_PHASES] - first, kDsMaxItems);
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_sched[DS_PHASES + 1 + i] = p.sched_items[first + i];
    const int words = p.L * (int)(sizeof(DsLayer) / 8);
    for (int i = threadIdx.x; i < words; i += blockDim.x)
      reinterpret_cast<unsigned long long*>(sbase + lay.layers)[i] = reinterpret_cast<const unsigned long long*>(p.layers)[i];
    if (threadIdx.x < (unsigned)p.T) {
      s_seq[threadIdx.x] = p.seq[threadIdx.x];
      s_pos[threadIdx.x] = p.pos[threadIdx.x];
    }
  }
  if (threadIdx.x < (unsigned)p.T) {  // the step's ids (async scheduling: gathered from the previous step)
    const int t = threadIdx.x;
    int id = p.ids[t];
    const int src = p.prev_row ? p.prev_row[t] : -1;
    if (src >= 0) id = src < p.prev_rows ? p.prev_ids[src] : -1;
    if (id < 0 || id >= p.V) {
      set_status(p.status, ST_NAN);
      id = 0;
    }
    s_ids[t] = id;
  }
  __syncthreads();
  if (threadIdx.x >= kDsConsumers) {
    if (threadIdx.x == kDsConsumers) ds_producer(p, S, epoch, &s_issued);
  } else {
    ds_consumer(p, S, epoch, &s_consumed);
  }
  __syncthreads();
  if (threadIdx.x == kDsConsumers) {
    // copies still in flight (a step given up) land before the CTA exits
    const uint32_t iss = s_issued, con = s_consumed;
    const uint32_t first = iss > (uint32_t)p.slots_n && iss - p.slots_n > con ? iss - p.slots_n : con;
    for (uint32_t q = first; q < iss; ++q) {
      const uint64_t t0 = global_ns();
      while (!mbar_try(&s_full[q % p.slots_n], (q / p.slots_n) & 1) && global_ns() - t0 < 1000ull * 1000 * 1000) {
      }
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.epoch, 1u);  // the next step's tags
  }
}

cudaError_t decode_step_prepare(size_t smem, int* max_ctas_per_sm) {
  const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(k_decode_step), (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_ctas_per_sm, k_decode_step, kDsThreads, smem);
}

cudaError_t launch_decode_step(const DecodeStepParams& p, int grid, size_t smem, cudaStream_t s) {
  if (p.T < 1 || p.T > p.trows || p.slots_n < 2 || p.slots_n > kDsMaxSlots) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: the phases wait on each other
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_step, p);
}

}  // namespace grd
