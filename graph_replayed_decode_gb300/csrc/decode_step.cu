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
static constexpr int kDsGroup = 3;   // 16-row tiles of one projection pass

// Word w (a pair of bf16 values) of a staged row is stored in MMA fragment order: inside each k-tile of 16
// words, the four words that lane quad q takes as its B fragments (q, q + 4, q + 8, q + 12) are adjacent, so
// one 16-byte shared load brings them.
__host__ __device__ constexpr int xperm(int w) { return (w & ~15) | ((w & 3) << 2) | ((w >> 2) & 3); }

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
// Non-blocking test of a phase (the common case: the ring chunk landed long ago).
ENG_DEVICE bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
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
  return mbar_test(bar, parity) || ds_mbar_spin(p, bar, parity, epoch, site);
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

// The attention overlay of the staging region: offsets of its buffers (16-byte aligned).
struct DsAttnOff {
  size_t qt, pt, abuf, sc, cs, kn, vn, mland, total;
};
__host__ __device__ inline size_t ds_up16(size_t x) { return (x + 15) & ~(size_t)15; }
__host__ __device__ inline DsAttnOff ds_attn_off(int d, int G) {
  const int kpc = 16 * ds_blocks_per_chunk(d);
  DsAttnOff o;
  size_t x = 0;
  o.qt = x;
  x += ds_up16((size_t)16 * (d + 8) * 2);
  o.pt = x;
  x += ds_up16((size_t)16 * (kpc + 8) * 2);
  o.abuf = x;
  x += ds_up16((size_t)10 * d * 4);
  o.sc = x;
  x += ds_up16((size_t)8 * kpc * 4);
  o.cs = x;
  x += ds_up16((size_t)3 * d * 4);
  o.kn = x;
  x += ds_up16((size_t)d * 2);
  o.vn = x;
  x += ds_up16((size_t)d * 2);
  o.mland = x;
  x += ds_up16((size_t)(kDsMaxSplits - 1) * G * (d + 2) * 4);
  o.total = x;
  return o;
}

// Shared memory of one CTA: the ring, the staging region (activation planes, or the attention overlay),
// the landing area of fetched word pairs (also the projection's partial tiles), the per-thread sums of
// squares, a stage's norm weights, the layer table and the schedule.
constexpr int kDsLandBytes = 8 * kDsConsumers * 8;
struct DsLayout {
  size_t ring, region, land, part, nwt, layers, sched, total;
};
__host__ __device__ inline DsLayout ds_layout(int slots_n, int trows, int kx, int d, int G, int H, int L) {
  DsLayout m;
  m.ring = 0;  // 1024-byte aligned at run time (the layout reserves the slack at the end)
  m.region = (size_t)slots_n * kDsSlotBytes;
  const size_t planes = (size_t)2 * trows * kx * 2, attn = ds_attn_off(d, G).total;
  m.land = m.region + ((planes > attn ? planes : attn) + 127) / 128 * 128;
  const size_t red = (size_t)kDsGroup * kDsWarps * 32 * 16;
  m.part = m.land + (red > (size_t)kDsLandBytes ? red : (size_t)kDsLandBytes);
  m.nwt = m.part + (size_t)trows * kDsConsumers * 4;
  m.layers = m.nwt + ds_up16((size_t)H * 4);
  m.sched = m.layers + ds_up16((size_t)L * sizeof(DsLayer));
  m.total = m.sched + (size_t)(DS_PHASES + 1 + kDsMaxItems) * 4 + 1024 + 128;
  return m;
}

size_t decode_step_smem(int slots_n, int trows, int kx, int d, int G, int H, int L) {
  return ds_layout(slots_n, trows, kx, d, G, H, L).total;
}

struct DsSmem {
  uint8_t* ring;
  bf16* xs;      // staged activation planes [trows][kx]
  bf16* xl;
  float4* red;   // [kDsGroup tiles][7 warps][32 lanes] partial tiles (aliases land)
  float* land;   // [8][kDsConsumers][2]: a fetch round's word pairs
  float* part;   // [trows][kDsConsumers] per-thread partial sums of squares
  float* nwt;    // [H] the norm weights of a stage
  // attention overlay of the staging region
  bf16* qt;      // [16][d + 8]: rows h = hi(q_h), 8 + h = lo(q_h)
  bf16* pt;      // [16][kpc + 8]: probabilities, hi and lo rows
  float* abuf;   // [(G + 2) d]: q heads, k, v of the token
  float* sc;     // [8][kpc] scores
  float* cs;     // [3 d]: cos/sin pairs of the token's position, then the q and k norm weights
  bf16* kn;      // [d] new key (bf16, roped)
  bf16* vn;      // [d] new value
  float* mland;  // [kDsMaxSplits - 1][G][d + 2]: the other splits' (O, max, sum), for the merge
  const DsLayer* layers;  // [L] weight pointers
  const int* off;         // [DS_PHASES + 1] this CTA's item ranges
  const int* items;       // this CTA's items
  const int* seq;         // [8] the rows' sequence lengths and positions
  const int* pos;
  uint64_t* full;
  uint64_t* empty;
  int* ids;      // [8]
  float* mrun;   // [8] online softmax state per head
  float* lrun;
  float* alpha;
  float* rs;     // [8] 1 / rms of the staged rows (norm phases)
};

// ------------------------------------------------------------------ producer: weights and K/V into the ring

struct DsChunk {
  const void* src[8];  // up to 8 copies (one weight range, or K and V blocks)
  uint32_t dst[8];     // offsets in the slot
  uint32_t bytes[8];
  int n;
};

// Attention item geometry shared by producer and consumer.  A row's keys are nch ring chunks (bpc blocks of
// 16 keys each), taken in order by its first na = min(NS, nch) splits of the step's NS, the first nch % na
// splits one chunk more than the others.  Split na - 1 holds the row's newest position (it writes the new
// K/V) and merges the others.  A padding row (length 0) has one split, which publishes a zero output.
struct DsAttnItem {
  int r, g, s, sl, nblk, na, c0, c1;
  bool merger, active;
};
// An attention item of the schedule is (r << 16) | (g << 8) | s.
ENG_DEVICE DsAttnItem ds_attn_item(const DecodeStepParams& p, const DsSmem& S, int item) {
  DsAttnItem a;
  const int NS = p.asplits;
  a.s = item & 255;
  a.g = (item >> 8) & 255;
  a.r = item >> 16;
  a.sl = S.seq[a.r];
  a.nblk = a.sl <= 0 ? 0 : min((a.sl + 15) >> 4, p.mbs);
  const int bpc_log2 = 31 - __clz(ds_blocks_per_chunk(p.d));  // blocks per chunk: a power of two
  const int nch = (a.nblk + (1 << bpc_log2) - 1) >> bpc_log2;
  a.na = max(1, min(NS, nch));
  a.active = a.s < a.na;
  a.merger = a.s == a.na - 1;
  // q chunks each, the first r splits one more (the merging split has the fewest); none past the active ones
  const int q = nch / a.na, r = nch - q * a.na;
  a.c0 = a.active ? a.s * q + min(a.s, r) : 0;
  a.c1 = a.active ? a.c0 + q + (a.s < r ? 1 : 0) : 0;
  return a;
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
#pragma unroll 1
  for (int l = 0; l < p.L; ++l) {
    const DsLayer& Lw = S.layers[l];
    // the LM head reads its weights right after this kernel: the first part of them into L2 while the last
    // layer runs (it leaves most of the memory bandwidth unused)
    if (l == p.L - 1 && p.pf_bytes) prefetch_share(p.pf_ptr, p.pf_bytes);
#pragma unroll 1
    for (int ph = 0; ph < DS_PHASES; ++ph) {
#pragma unroll 1
      for (int it = off[ph]; it < off[ph + 1]; ++it) {
        const int item = S.items[it];
        int nch;
        DsAttnItem a;
        const bf16* W = nullptr;
        int KT = 0;
        if (ph == DS_ATTN) {
          a = ds_attn_item(p, S, item);
          nch = a.c1 - a.c0;
        } else {
          const int K = ph == DS_O ? p.Hq * p.d : ph == DS_DOWN ? p.I : p.H;
          W = ph == DS_QKV ? Lw.qkv : ph == DS_O ? Lw.o : ph == DS_GU ? Lw.gu : Lw.down;
          KT = K >> 5;
          nch = (KT + 31) >> 5;
        }
#pragma unroll 1
        for (int c = 0; c < nch; ++c, ++q, rp.next(NS)) {
          const int slot = rp.slot;
          if (rp.round > 0 && !ds_mbar_wait(p, &S.empty[slot], (rp.round - 1) & 1, epoch, WAIT_RING_EMPTY)) {
            *issued_out = q;
            return;
          }
          uint8_t* dst = S.ring + (size_t)slot * kDsSlotBytes;
          if (ph == DS_ATTN) {
            const int bb = (a.c0 + c) * bpc, be = max(bb, min(a.nblk, bb + bpc));  // never a negative count
            mbar_expect_tx(&S.full[slot], (uint32_t)(be - bb) * 2u * blk_bytes);
#pragma unroll 1
            for (int b = bb; b < be; ++b) {
              int blk = p.bt[(size_t)a.r * p.mbs + b];
              if (blk < 0 || blk >= p.NB) blk = p.NB;  // flagged by the consumer; the scratch block is harmless
#pragma unroll 1
              for (int kv = 0; kv < 2; ++kv) {
                const int row0 = (int)(((((size_t)l * 2 + kv) * (p.NB + 1) + blk) * p.Hkv + a.g) * 16);
                uint8_t* bd = dst + (size_t)kv * bpc * blk_bytes + (size_t)(b - bb) * blk_bytes;
#pragma unroll 1
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

// Tag of the words of layer l's phase ph in the step of this epoch; layer -1's DOWN phase (tag value 0 in
// the low byte) is the step's embedding rows, which the kernel's prologue writes.
ENG_DEVICE uint32_t ds_tag(uint32_t epoch, int l, int ph) { return (epoch << 8) | (uint32_t)(l * DS_PHASES + ph + 1); }

// Up to three runs of tagged word pairs to fetch into shared memory as floats: pair i of run r is the words
// src_r[2i], src_r[2i + 1]; the runs are taken in order.
struct DsRuns {
  const unsigned long long *src0, *src1, *src2;
  float *dst0, *dst1, *dst2;
  int n0, n1, n2;  // pairs of each run
};

// One round of a fetch: the pairs [base, base + 8 kDsConsumers) of the runs' concatenation, this thread taking
// pairs base + tid + j kDsConsumers.  All of them are requested at once, the ones still without the tag are
// requested again together, and each pair lands in its run's dst (at 2i), or in `land` at
// 2 (pair - base) when land is given.  Returns false when the step is given up.
ENG_DEVICE bool ds_fetch(const DecodeStepParams& p, const DsRuns& R, int base, float* land, uint32_t tag,
                         uint32_t epoch, int site) {
  const int tid = threadIdx.x;
  const int e0 = R.n0, e1 = e0 + R.n1, e2 = e1 + R.n2;
  unsigned long long a[8][2];
  unsigned have = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int pi = base + tid + j * kDsConsumers;
    if (pi < e2) {
      const unsigned long long* at = pi < e0 ? R.src0 + 2 * pi : pi < e1 ? R.src1 + 2 * (pi - e0) : R.src2 + 2 * (pi - e1);
      ll_load2(at, a[j][0], a[j][1]);
      have |= 1u << j;
    }
  }
  unsigned pending = have;
  DsWait wt = ds_wait(epoch, site);
  while (true) {
    unsigned still = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (ll_tag(a[j][0]) != tag || ll_tag(a[j][1]) != tag) still |= 1u << j;
    still &= pending;
    if (!still) break;
    if (!ds_keep_waiting(p, wt)) return false;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((still >> j) & 1u) {
        const int pi = base + tid + j * kDsConsumers;
        const unsigned long long* at = pi < e0 ? R.src0 + 2 * pi : pi < e1 ? R.src1 + 2 * (pi - e0) : R.src2 + 2 * (pi - e1);
        ll_load2(at, a[j][0], a[j][1]);
      }
    pending = still;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if ((have >> j) & 1u) {
      const int pi = base + tid + j * kDsConsumers;
      float* dst = land ? land + 2 * (pi - base) : pi < e0 ? R.dst0 + 2 * pi : pi < e1 ? R.dst1 + 2 * (pi - e0) : R.dst2 + 2 * (pi - e1);
      *reinterpret_cast<float2*>(dst) = make_float2(ll_val(a[j][0]), ll_val(a[j][1]));
    }
  return true;
}

// Stages the T rows of width K of a tagged vector as the hi/lo planes of x * w (w == nullptr: x itself) in
// fragment order, and leaves each thread's partial sums of squares of every row in S.part (ds_rms adds them
// up).  Up to 8 word pairs per thread are requested at once, with their norm weights; the pairs still
// without the tag are requested again together.
ENG_DEVICE bool ds_stage(const DecodeStepParams& p, const DsSmem& S, const unsigned long long* src, uint32_t tag,
                         int K, const float* w, uint32_t epoch) {
  const int tid = threadIdx.x;
#pragma unroll 1
  for (int t = 0; t < p.T; ++t) S.part[t * kDsConsumers + tid] = 0.f;
  int cur = -1;
  float run = 0.f;
  bool ok = true;
  const int npairs = p.T * K / 2;
#pragma unroll 1
  for (int base = tid; base < npairs && ok; base += kDsConsumers * 8) {
    const int t0 = (2 * base) / K, c0 = 2 * base - t0 * K;  // row and column of this round's first pair
    unsigned long long a[8][2];
    float2 wv[8];
    unsigned pending = 0;
    {
      int c = c0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int pi = base + j * kDsConsumers;
        if (pi < npairs) {
          ll_load2(src + 2 * pi, a[j][0], a[j][1]);
          wv[j] = w ? make_float2(__ldg(w + c), __ldg(w + c + 1)) : make_float2(1.f, 1.f);
          pending |= 1u << j;
        }
        c += 2 * kDsConsumers;
        while (c >= K) c -= K;
      }
    }
    DsWait wt = ds_wait(epoch, WAIT_STAGE);
    while (true) {
      unsigned still = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (ll_tag(a[j][0]) != tag || ll_tag(a[j][1]) != tag) still |= 1u << j;
      still &= pending;
      if (!still) break;
      if (!ds_keep_waiting(p, wt)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if ((still >> j) & 1u) ll_load2(src + 2 * (base + j * kDsConsumers), a[j][0], a[j][1]);
      pending = still;
    }
    if (!ok) break;
    int t = t0, c = c0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (base + j * kDsConsumers >= npairs) break;
      const float v0 = ll_val(a[j][0]), v1 = ll_val(a[j][1]);
      uint32_t h, lo;
      split_bf16x2(v0 * wv[j].x, v1 * wv[j].y, h, lo);
      const int wi = t * (p.kx >> 1) + xperm(c >> 1);
      reinterpret_cast<uint32_t*>(S.xs)[wi] = h;
      reinterpret_cast<uint32_t*>(S.xl)[wi] = lo;
      if (t != cur) {  // each thread's pairs of a row are consecutive in its walk
        if (cur >= 0) S.part[cur * kDsConsumers + tid] = run;
        cur = t;
        run = 0.f;
      }
      run += v0 * v0 + v1 * v1;
      c += 2 * kDsConsumers;
      while (c >= K) {
        c -= K;
        ++t;
      }
    }
  }
  if (cur >= 0) S.part[cur * kDsConsumers + tid] = run;
  return csync_and(ok);
}

// Row t's sum of squares from the stage's per-thread parts, by one warp: the parts in thread order within
// each warp's lanes, the warps' sums by a fixed xor tree.
ENG_DEVICE float ds_sumsq(const DsSmem& S, int t) {
  const int lane = threadIdx.x & 31;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kDsWarps; ++j) ss += S.part[t * kDsConsumers + lane + 32 * j];
  return warp_sum(ss);
}

// The LM head's inputs after the final stage (every word of h is known to carry its tag): the final residual
// rows and the planes of h * final norm weight, in row-major order.
ENG_DEVICE void ds_final_rows(const DecodeStepParams& p, const DsSmem& S, const unsigned long long* h) {
  const int warp = threadIdx.x >> 5;
#pragma unroll 1
  for (int t = warp; t < p.T; t += kDsWarps) {
    const float ss = ds_sumsq(S, t);
    if ((threadIdx.x & 31) == 0) p.sq[(size_t)t * p.sq_stride] = ss;
  }
#pragma unroll 1
  for (int i = 2 * threadIdx.x; i < p.T * p.H; i += 2 * kDsConsumers) {
    unsigned long long a, b;
    ll_load2(h + i, a, b);
    const int c = i % p.H;
    p.h_out[i] = ll_val(a);
    p.h_out[i + 1] = ll_val(b);
    put_split2(p.xn_h, p.xn_l, (size_t)i, ll_val(a) * __ldg(p.final_norm + c), ll_val(b) * __ldg(p.final_norm + c + 1));
  }
}

// This token's q heads, k and v of one KV head from the QKV phase's words into S.abuf [(G + 2) d] (fp32).
ENG_DEVICE bool ds_gather_head(const DecodeStepParams& p, const DsSmem& S, const unsigned long long* qrow, int g,
                               uint32_t tag, uint32_t epoch) {
  const int d = p.d, G = p.Hq / p.Hkv;
  const DsRuns R{qrow + (size_t)g * G * d, qrow + (size_t)(p.Hq + g) * d, qrow + (size_t)(p.Hq + p.Hkv + g) * d,
                 S.abuf, S.abuf + G * d, S.abuf + (G + 1) * d, G * d / 2, d / 2, d / 2};
  bool ok = true;
#pragma unroll 1
  for (int base = 0; base < (G + 2) * d / 2 && ok; base += 8 * kDsConsumers)
    ok = ds_fetch(p, R, base, nullptr, tag, epoch, WAIT_HEAD);
  return ok;
}

// The n (<= kDsGroup) 16-row tiles of a packed weight ([N][K]) that one pass of a projection phase takes,
// against the staged planes.  In each ring chunk warp w takes the k-tiles w, w + 7, ... into four independent
// accumulator chains of its tile (two k-steps x hi/lo planes); tiles of a single chunk each (K <= 1024) run
// interleaved, the chunks of all n tiles being in the ring together.  The warps' sums are added in warp
// order.  On return warp i (< n) holds tile i's values in v, in MMA fragment order: (row r, token c),
// (r, c + 1), (r + 8, c), (r + 8, c + 1) with r = lane / 4, c = 2 (lane % 4); with `norm`, rs holds
// 1 / rms of the staged rows c and c + 1 (ds_stage's parts).  A row past the step's tokens reads row 0, so
// lanes of one step's rows read the same words as a broadcast.
ENG_DEVICE bool ds_gemv(const DecodeStepParams& p, const DsSmem& S, int K, int n, bool norm, RingPos& rp,
                        uint32_t epoch, float4& v, float (&rs)[2]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KT = K >> 5, nch = (KT + 31) >> 5;
  const int g = lane >> 2;
  const int xrow = g < p.T ? g : 0;
  const uint4* xs = reinterpret_cast<const uint4*>(S.xs + (size_t)xrow * p.kx) + (lane & 3);
  const uint4* xl = reinterpret_cast<const uint4*>(S.xl + (size_t)xrow * p.kx) + (lane & 3);
  // 1 / rms of the staged rows, by the last warp (it has the fewest k-tiles) before its MMA pass; the
  // reduction's barrier below publishes it to the epilogue warps
  if (norm && warp == kDsWarps - 1) {
#pragma unroll 1
    for (int t = 0; t < p.T; ++t) {
      const float r_t = rsqrtf(ds_sumsq(S, t) / (float)K + p.eps);
      if (lane == 0) S.rs[t] = r_t;
    }
  }
  bool ok = true;
  if (nch == 1 && n <= p.slots_n) {  // every tile's chunk fits in the ring at once
    float acc[kDsGroup][4][4];
#pragma unroll
    for (int i = 0; i < kDsGroup; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
    RingPos r2 = rp;
    const uint4* w[kDsGroup];
#pragma unroll
    for (int i = 0; i < kDsGroup; ++i) {
      w[i] = reinterpret_cast<const uint4*>(S.ring + (size_t)r2.slot * kDsSlotBytes) + lane;
      if (i < n) {
        if (ok && !ds_mbar_wait(p, &S.full[r2.slot], r2.round & 1, epoch)) ok = false;
        r2.next(p.slots_n);
      }
    }
    if (ok) {
#pragma unroll
      for (int j = 0; j < (32 + kDsWarps - 1) / kDsWarps; ++j) {
        const int kt = warp + kDsWarps * j;
        if (kt >= KT) break;
        const uint4 bh = xs[kt * 4], bl = xl[kt * 4];
#pragma unroll
        for (int i = 0; i < kDsGroup; ++i) {
          if (i >= n) break;
          const uint4 a0 = w[i][kt * 64], a1 = w[i][kt * 64 + 32];
          mma_bf16(acc[i][0], a0.x, a0.y, a0.z, a0.w, bh.x, bh.y);
          mma_bf16(acc[i][1], a1.x, a1.y, a1.z, a1.w, bh.z, bh.w);
          mma_bf16(acc[i][2], a0.x, a0.y, a0.z, a0.w, bl.x, bl.y);
          mma_bf16(acc[i][3], a1.x, a1.y, a1.z, a1.w, bl.z, bl.w);
        }
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < kDsGroup; ++i) {
        if (i >= n) break;
        if (lane == 0) mbar_arrive(&S.empty[rp.slot]);
        rp.next(p.slots_n);
        S.red[(i * kDsWarps + warp) * 32 + lane] =
            make_float4((acc[i][0][0] + acc[i][1][0]) + (acc[i][2][0] + acc[i][3][0]),
                        (acc[i][0][1] + acc[i][1][1]) + (acc[i][2][1] + acc[i][3][1]),
                        (acc[i][0][2] + acc[i][1][2]) + (acc[i][2][2] + acc[i][3][2]),
                        (acc[i][0][3] + acc[i][1][3]) + (acc[i][2][3] + acc[i][3][3]));
      }
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < n && ok; ++i) {
      float acc[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll 1
      for (int c = 0; c < nch; ++c, rp.next(p.slots_n)) {
        if (!ds_mbar_wait(p, &S.full[rp.slot], rp.round & 1, epoch)) {
          ok = false;
          break;
        }
        const uint4* w = reinterpret_cast<const uint4*>(S.ring + (size_t)rp.slot * kDsSlotBytes) + lane;
        const int nkt = min(32, KT - 32 * c);
        const uint4* xsc = xs + 32 * c * 4;
        const uint4* xlc = xl + 32 * c * 4;
#pragma unroll
        for (int j = 0; j < (32 + kDsWarps - 1) / kDsWarps; ++j) {
          const int kt = warp + kDsWarps * j;
          if (kt >= nkt) break;
          const uint4 a0 = w[kt * 64], a1 = w[kt * 64 + 32];
          const uint4 bh = xsc[kt * 4], bl = xlc[kt * 4];
          mma_bf16(acc[0], a0.x, a0.y, a0.z, a0.w, bh.x, bh.y);
          mma_bf16(acc[1], a1.x, a1.y, a1.z, a1.w, bh.z, bh.w);
          mma_bf16(acc[2], a0.x, a0.y, a0.z, a0.w, bl.x, bl.y);
          mma_bf16(acc[3], a1.x, a1.y, a1.z, a1.w, bl.z, bl.w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[rp.slot]);
      }
      S.red[(i * kDsWarps + warp) * 32 + lane] =
          make_float4((acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]), (acc[0][1] + acc[1][1]) + (acc[2][1] + acc[3][1]),
                      (acc[0][2] + acc[1][2]) + (acc[2][2] + acc[3][2]), (acc[0][3] + acc[1][3]) + (acc[2][3] + acc[3][3]));
    }
  }
  if (!csync_and(ok)) return false;
  if (warp < n) {
    const float4* r = S.red + (size_t)warp * kDsWarps * 32 + lane;
    float4 u[kDsWarps];
#pragma unroll
    for (int w2 = 0; w2 < kDsWarps; ++w2) u[w2] = r[w2 * 32];
    const int c = 2 * (lane & 3);
    rs[0] = norm && c < p.T ? S.rs[c] : 1.f;
    rs[1] = norm && c + 1 < p.T ? S.rs[c + 1] : 1.f;
    v = u[0];
#pragma unroll
    for (int w2 = 1; w2 < kDsWarps; ++w2) {
      v.x += u[w2].x;
      v.y += u[w2].y;
      v.z += u[w2].z;
      v.w += u[w2].w;
    }
  }
  return true;
}

// Attention of one item: request row r, KV head g, key split s.  QK-norm and RoPE of the token's q heads
// and k, the write of the new K/V (by the last split, which holds the new position), online softmax over
// the item's chunks, then either this split's (O, max, sum) as tagged words or, in the last split, the merge
// of the row's splits in split order into the attention output words.
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
  if (tid == 0 && a.merger && a.g == 0 && a.sl > 0 && (!pos_ok || ((a.sl + 15) >> 4) > p.mbs))
    set_status(p.status, ST_BAD_POSITION);

  // ---- the RoPE row and the QK-norm weights into shared memory (asynchronous copies, waited for below)
  const DsLayer& Lw = S.layers[l];
  const bool qk_norm = Lw.q_norm != nullptr;
  if (tid < 3 * (d / 4)) {
    const int sh = 29 - __clz(d);  // log2(d / 4)
    const int arr = tid >> sh, piece = tid & ((d >> 2) - 1);
    const float* src = arr == 0 ? p.rope + (size_t)pos * d : arr == 1 ? Lw.q_norm : Lw.k_norm;
    if (src) cp_async16(S.cs + arr * d + 4 * piece, src + 4 * piece);
  }
  cp_async_commit();
  // ---- this token's q heads, k and v
  // the block that takes the new position (the last split writes it), requested before the gather
  const int new_blk = a.merger && a.sl > 0 && pos_ok ? __ldg(p.bt + (size_t)a.r * p.mbs + (pos >> 4)) : -1;
  // (the q and probability tiles' rows past the heads are not cleared: each MMA row feeds only its own
  // output row, and those rows are never read)
  bool ok = ds_gather_head(p, S, qrow, a.g, tag_in, epoch);
  if (tid < 8) {
    S.mrun[tid] = -INFINITY;
    S.lrun[tid] = 0.f;
  }
  cp_async_wait<0>();
  if (!csync_and(ok)) return false;

  // ---- QK-norm and rotate-half RoPE (warp per head row: q heads, then k); v is only rounded
#pragma unroll 1
  for (int row = warp; row < G + 2; row += kDsWarps) {
    float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < E) x[e] = S.abuf[row * d + lane * E + e];
    if (row <= G) {
      if (qk_norm) {
        const float* nw = S.cs + (row < G ? d : 2 * d);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) ss += x[e] * x[e];
        ss = warp_sum(ss);
        const float rs = rsqrtf(ss / (float)d + p.eps);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < E) x[e] = x[e] * rs * nw[lane * E + e];
      }
      float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
        const int ii = (lane & 15) * E + e;
        if (e < E) {
          const float c = S.cs[2 * ii], sn = S.cs[2 * ii + 1];
          y[e] = (lane < 16) ? (x[e] * c - other * sn) : (x[e] * c + other * sn);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = y[e];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e >= E) break;
      const bf16 h = __float2bfloat16_rn(x[e]);
      if (row < G) {
        S.qt[row * (d + 8) + lane * E + e] = h;
        S.qt[(8 + row) * (d + 8) + lane * E + e] = __float2bfloat16_rn(x[e] - __bfloat162float(h));
      } else {
        (row == G ? S.kn : S.vn)[lane * E + e] = h;
      }
    }
  }
  csync();

  // ---- the new K/V into the paged pool (the last split holds the new position; padding: scratch block)
  if (a.merger) {
    int slot = -1;
    if (a.sl > 0) {
      if (!pos_ok) {
        slot = -2;
      } else {
        slot = (new_blk < 0 || new_blk >= p.NB) ? -3 : new_blk * 16 + (pos & 15);
      }
    }
    const int blk = slot >= 0 ? slot >> 4 : p.NB, off = slot >= 0 ? slot & 15 : 0;
    const size_t o = (((size_t)blk * p.Hkv + a.g) * 16 + off) * d;
    bf16* kp = const_cast<bf16*>(ds_plane(p, l, 0)) + o;
    bf16* vp = const_cast<bf16*>(ds_plane(p, l, 1)) + o;
#pragma unroll 1
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
  unsigned long long* out = p.attn_out + (size_t)t * p.Hq * d + (size_t)a.g * G * d;      // [G][d]
  if (a.sl <= 0) {  // a padding row attends to nothing: a zero output
#pragma unroll 1
    for (int i = tid; i < G * d; i += kDsConsumers) ll_store(out + i, 0.f, tag_out);
    return true;
  }

  // ---- online softmax over the item's chunks (base 2)
  const int gl = lane >> 2, tl = lane & 3;  // MMA fragment row group and column pair of this lane
  const int nd = d / 8;                     // 8-column tiles of the output
  constexpr int kOt = (16 + kDsWarps - 1) / kDsWarps;  // output column tiles per warp (d / 8 <= 16)
  float o[kOt][4];
#pragma unroll
  for (int j = 0; j < kOt; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  const int nch = a.c1 - a.c0;
  const uint32_t blk_bytes = 16u * d * 2u;
#pragma unroll 1
  for (int c = 0; c < nch; ++c, rp.next(p.slots_n), ++q) {
    const int slot = rp.slot;
    if (!ds_mbar_wait(p, &S.full[slot], rp.round & 1, epoch)) ok = false;
    if (!csync_and(ok)) return false;
    bf16* Kc = reinterpret_cast<bf16*>(S.ring + (size_t)slot * kDsSlotBytes);
    bf16* Vc = reinterpret_cast<bf16*>(S.ring + (size_t)slot * kDsSlotBytes + (size_t)bpc * blk_bytes);
    const int bb = (a.c0 + c) * bpc, nb = min(a.nblk, bb + bpc) - bb;
    const int key0 = bb * 16, kb = nb * 16;
    // the new position's key and value (the pool copy may predate this step), and zero values for keys
    // past the row's length (a freed block's stale contents must not reach the product)
    uint8_t* Kb = reinterpret_cast<uint8_t*>(Kc);
    uint8_t* Vb = reinterpret_cast<uint8_t*>(Vc);
    const int kvalid = min(kb, a.sl - key0);
    if ((pos >= key0 && pos < key0 + kb) || kvalid < kb) {
      if (pos >= key0 && pos < key0 + kb && tid < d / 4) {  // one 16-byte chunk of K or V per thread
        const int cc = tid % (d / 8);
        uint8_t* dstc = (tid < d / 8 ? Kb : Vb) + kv_off(pos - key0, cc, blk_bytes);
        *reinterpret_cast<uint4*>(dstc) = reinterpret_cast<const uint4*>(tid < d / 8 ? S.kn : S.vn)[cc];
      }
#pragma unroll 1
      for (int i = tid; i < (kb - kvalid) * (d / 8); i += kDsConsumers)
        *reinterpret_cast<uint4*>(Vb + kv_off(kvalid + i / (d / 8), i % (d / 8), blk_bytes)) = make_uint4(0u, 0u, 0u, 0u);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes before the slot's next copy
      csync();
    }

    // S = Q K^T: warp w takes the 8-key tiles w, w + 8
#pragma unroll 1
    for (int nt = warp; nt < kb / 8; nt += kDsWarps) {
      float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sodd[4] = {0.f, 0.f, 0.f, 0.f};  // even and odd k-steps
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int ks = 2 * kk;
        if (ks >= d / 16) break;
        uint32_t af[4], af2[4], bfr[4];
        ldmatrix_x4(af, S.qt + (size_t)(lane & 15) * (d + 8) + ks * 16 + (lane >> 4) * 8);
        ldmatrix_x4(af2, S.qt + (size_t)(lane & 15) * (d + 8) + (ks + 1) * 16 + (lane >> 4) * 8);
        ldmatrix_x4(bfr, Kb + kv_off(nt * 8 + (lane & 7), 2 * ks + (lane >> 3), blk_bytes));
        mma_bf16(sacc, af[0], af[1], af[2], af[3], bfr[0], bfr[1]);
        mma_bf16(sodd, af2[0], af2[1], af2[2], af2[3], bfr[2], bfr[3]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[e] += sodd[e];
      if (gl < G) {
        const int k = nt * 8 + 2 * tl;
        const float s0 = (sacc[0] + sacc[2]) * p.scale_log2, s1 = (sacc[1] + sacc[3]) * p.scale_log2;
        S.sc[gl * kpc + k] = key0 + k < a.sl ? s0 : -INFINITY;
        S.sc[gl * kpc + k + 1] = key0 + k + 1 < a.sl ? s1 : -INFINITY;
      }
    }
    csync();
    // per head (a warp each): the chunk's maximum, the probabilities as hi/lo rows, the running sum
#pragma unroll 1
    for (int hh = warp; hh < G; hh += kDsWarps) {
      float mx = -INFINITY;
#pragma unroll 1
      for (int k = lane; k < kb; k += 32) mx = fmaxf(mx, S.sc[hh * kpc + k]);
      mx = warp_max(mx);
      const float m_old = S.mrun[hh], m_new = fmaxf(m_old, mx);
      float sum = 0.f;
#pragma unroll 1
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
#pragma unroll 4
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

  if (!a.merger) {
    // ---- this split's (O unnormalised, running max, running sum) as tagged words for the row's last split
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
  // ---- the last split merges the row's splits in split order: M = the largest max, w_s = 2^(max_s - M),
  // out = (sum_s w_s O_s) / (sum_s w_s sum_s); its own (O, max, sum) come from registers and shared memory
  float* own = S.abuf;  // [G][d]
  if (gl < G) {
#pragma unroll
    for (int j = 0; j < kOt; ++j) {
      const int ndt = warp + kDsWarps * j;
      if (ndt >= nd) continue;
      own[gl * d + ndt * 8 + 2 * tl] = o[j][0] + o[j][2];
      own[gl * d + ndt * 8 + 2 * tl + 1] = o[j][1] + o[j][3];
    }
  }
  // the other splits' words (splits 0 .. na - 2 are contiguous in the workspace)
  const int npm = (a.na - 1) * G * (int)wrow / 2;
  const DsRuns R{ws, nullptr, nullptr, S.mland, nullptr, nullptr, npm, 0, 0};
#pragma unroll 1
  for (int base = 0; base < npm && ok; base += 8 * kDsConsumers)
    ok = ds_fetch(p, R, base, nullptr, tag_out, epoch, WAIT_ATTN_MERGE);
  if (!csync_and(ok)) return false;

  // per head (a warp each): M = the largest max, f_s = 2^(max_s - M) / sum_s' 2^(max_s' - M) sum_s'
  float* f = S.sc;  // [na][G]
#pragma unroll 1
  for (int h = warp; h < G; h += kDsWarps) {
    const int sp = lane;  // split of this lane (the last split: the merger's own)
    float m = -INFINITY, lsum = 0.f;
    if (sp < a.na - 1) {
      m = S.mland[((size_t)sp * G + h) * wrow + d];
      lsum = S.mland[((size_t)sp * G + h) * wrow + d + 1];
    } else if (sp == a.na - 1) {
      m = S.mrun[h];
      lsum = S.lrun[h];
    }
    const float M = warp_max(m);
    const float wgt = sp < a.na ? exp2f(m - M) : 0.f;
    const float L = warp_sum(wgt * lsum);
    if (sp < a.na) f[sp * G + h] = wgt / L;
  }
  csync();
#pragma unroll 1
  for (int e2 = tid; e2 < G * d / 2; e2 += kDsConsumers) {  // element pairs: one pass for G * d <= 448
    const int e = 2 * e2, h = e / d;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
    for (int sp = 0; sp < a.na - 1; ++sp) {
      const float fs = f[sp * G + h];
      const float2 m2 = *reinterpret_cast<const float2*>(S.mland + ((size_t)sp * G + h) * wrow + (e - h * d));
      a0 += fs * m2.x;
      a1 += fs * m2.y;
    }
    const float fo = f[(a.na - 1) * G + h];
    a0 += fo * own[e];
    a1 += fo * own[e + 1];
    ll_store(out + e, a0, tag_out);
    ll_store(out + e + 1, a1, tag_out);
  }
  return true;
}

// Epilogue of one tile of a projection phase, by one warp whose lanes hold four values of the tile each
// (rows r, r + 8 and tokens c, c + 1 with r = lane / 4, c = 2 (lane % 4); ds_gemv):
//   QKV   the raw projection, 1 / rms of the input applied (rs: tokens c, c + 1), + bias (bias[k]: row r + 8 k);
//   O     h = h_prev (the previous layer's output, or the embedding in layer 0) + the tile;
//   GU    silu(gate) * up: tile rows 0..7 are gate rows and rows 8..15 the matching up rows;
//   DOWN  h = h after O + the tile.
// res[k]: the residual word of (row r + 8 (k / 2), token c + k % 2), requested before the product.
ENG_DEVICE bool ds_epilogue(const DecodeStepParams& p, int ph, int tile, const unsigned long long (&res)[4],
                            const float (&bias)[2], const float (&rs)[2], uint32_t tres, uint32_t tout, uint32_t epoch,
                            const float4& v) {
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, c = 2 * (lane & 3);
  const float val[4] = {v.x, v.y, v.z, v.w};
  if (ph == DS_GU) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = c + k;
      if (t >= p.T) break;
      const float ga = val[k] * rs[k], up = val[2 + k] * rs[k];
      ll_store(p.act_ll + (size_t)t * p.I + tile * 8 + r, ga / (1.f + expf(-ga)) * up, tout);
    }
    return true;
  }
  if (ph == DS_QKV) {
    const int QKV = (p.Hq + 2 * p.Hkv) * p.d;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = c + (k & 1);
      if (t < p.T)
        ll_store(p.qkv_ll + (size_t)t * QKV + tile * 16 + r + 8 * (k >> 1), val[k] * rs[k & 1] + bias[k >> 1], tout);
    }
    return true;
  }
  unsigned long long wd[4] = {res[0], res[1], res[2], res[3]};
  DsWait wt = ds_wait(epoch, WAIT_RESIDUAL);
  while (true) {
    unsigned still = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (c + (k & 1) < p.T && ll_tag(wd[k]) != tres) still |= 1u << k;
    if (!still) break;
    if (!ds_keep_waiting(p, wt)) return false;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if ((still >> k) & 1u) wd[k] = ll_load1(p.h_ll + (size_t)(c + (k & 1)) * p.H + tile * 16 + r + 8 * (k >> 1));
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int t = c + (k & 1);
    if (t < p.T) ll_store(p.h_ll + (size_t)t * p.H + tile * 16 + r + 8 * (k >> 1), ll_val(wd[k]) + val[k], tout);
  }
  return true;
}

// The consumer warps: every (layer, phase) of the step in order, then -- in CTA 0 -- the LM head's inputs.
// Each code path has a single call site, so that a layer runs through little code.
ENG_DEVICE void ds_consumer(const DecodeStepParams& p, const DsSmem& S, uint32_t epoch, uint32_t* consumed) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  RingPos rp{0, 0};
  uint32_t q = 0;  // chunks consumed
  bool ok = true;
  const int steps = p.L * DS_PHASES;
#pragma unroll 1
  for (int step = 0; step <= steps && ok; ++step) {
    const bool fin = step == steps;  // the final residual for the LM head (CTA 0)
    if (fin && blockIdx.x != 0) break;
    const int l = fin ? p.L - 1 : step / DS_PHASES, ph = fin ? DS_DOWN : step % DS_PHASES;
    const DsLayer& Lw = S.layers[l];
    if (tid == 0 && blockIdx.x < 1024) {
      g_ds_layer[blockIdx.x] = l;
      g_ds_phase[blockIdx.x] = ph;
    }
    const int first = fin ? 0 : S.off[ph], last = fin ? 0 : S.off[ph + 1];
    if (ph == DS_ATTN) {
#pragma unroll 1
      for (int it = first; ok && it < last; ++it)
        ok = ds_attention(p, S, l, S.items[it], rp, q, ds_tag(epoch, l, DS_QKV), ds_tag(epoch, l, DS_ATTN), epoch);
    } else if (first < last || fin) {
      // the phase's input rows, and for O and DOWN the tag of the residual they add to (h_ll)
      const unsigned long long* src = p.h_ll;
      uint32_t tag = ds_tag(epoch, l, DS_O);
      int K = p.H;
      bool norm = true;
      const float* w = Lw.post_norm;
      uint32_t tres = ds_tag(epoch, l, DS_O);
      if (fin) {
        tag = ds_tag(epoch, l, DS_DOWN);
        w = p.final_norm;
      } else if (ph == DS_QKV) {
        tag = ds_tag(epoch, l - 1, DS_DOWN);  // layer 0: the embedding rows
        w = Lw.in_norm;
      } else if (ph == DS_O) {
        src = p.attn_out;
        tag = ds_tag(epoch, l, DS_ATTN);
        K = p.Hq * p.d;
        w = nullptr;
        norm = false;
        tres = ds_tag(epoch, l - 1, DS_DOWN);
      } else if (ph == DS_DOWN) {
        src = p.act_ll;
        tag = ds_tag(epoch, l, DS_GU);
        K = p.I;
        w = nullptr;
        norm = false;
      }
      const bool resid = ph == DS_O || ph == DS_DOWN;
      // warp i finishes tile i of a group: its residual words and bias, requested before the inputs are
      // staged (the first group) or the product runs, so that they overlap the wait
      unsigned long long pre[4] = {0ull, 0ull, 0ull, 0ull};
      float bias[2] = {0.f, 0.f};
      auto request = [&](int it) {
        const int n = min(kDsGroup, last - it);
        if (warp >= n) return;
        const int tile = S.items[it + warp];
        if (resid) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int t = 2 * (lane & 3) + (k & 1), row = tile * 16 + (lane >> 2) + 8 * (k >> 1);
            if (t < p.T) pre[k] = ll_load1(p.h_ll + (size_t)t * p.H + row);
          }
        }
        if (ph == DS_QKV && Lw.qkv_bias) {
          bias[0] = __ldg(Lw.qkv_bias + tile * 16 + (lane >> 2));
          bias[1] = __ldg(Lw.qkv_bias + tile * 16 + (lane >> 2) + 8);
        }
      };
      if (first < last) request(first);
      ok = ds_stage(p, S, src, tag, K, w, epoch);
      if (ok && fin) ds_final_rows(p, S, src);
#pragma unroll 1
      for (int it = first; ok && it < last; it += kDsGroup) {
        const int n = min(kDsGroup, last - it);
        const int tile = warp < n ? S.items[it + warp] : 0;
        if (it != first) request(it);
        const uint32_t nch = (uint32_t)((K / 32 + 31) / 32);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        float rs[2] = {1.f, 1.f};  // 1 / rms of the lane's tokens c, c + 1 (norm phases)
        ok = ds_gemv(p, S, K, n, norm, rp, epoch, v, rs);
        ok = ok && csync_and(warp >= n || ds_epilogue(p, ph, tile, pre, bias, rs, tres, ds_tag(epoch, l, ph), epoch, v));
        q += (uint32_t)n * nch;
      }
    }
    if (ph == DS_DOWN) ok = csync_and(ok);
  }
  if (tid == 0) *consumed = q;
}

__global__ void __launch_bounds__(kDsThreads, 1) k_decode_step(const __grid_constant__ DecodeStepParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t s_full[kDsMaxSlots], s_empty[kDsMaxSlots];
  __shared__ float s_m[8], s_l[8], s_alpha[8], s_rs[8];
  __shared__ int s_ids[8], s_seq[8], s_pos[8];
  __shared__ uint32_t s_issued, s_consumed;
  const int G = p.Hq / p.Hkv;
  const DsLayout lay = ds_layout(p.slots_n, p.trows, p.kx, p.d, G, p.H, p.L);
  DsSmem S;
  // every region at a fixed offset from a 1024-byte aligned base (the swizzled tensor copies need it)
  uint8_t* const sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem) + 1023) & ~static_cast<uintptr_t>(1023));
  S.ring = sbase + lay.ring;
  S.xs = reinterpret_cast<bf16*>(sbase + lay.region);
  S.xl = S.xs + (size_t)p.trows * p.kx;
  S.red = reinterpret_cast<float4*>(sbase + lay.land);
  S.land = reinterpret_cast<float*>(sbase + lay.land);
  S.part = reinterpret_cast<float*>(sbase + lay.part);
  S.nwt = reinterpret_cast<float*>(sbase + lay.nwt);
  {
    const DsAttnOff ao = ds_attn_off(p.d, G);
    uint8_t* o = sbase + lay.region;
    S.qt = reinterpret_cast<bf16*>(o + ao.qt);
    S.pt = reinterpret_cast<bf16*>(o + ao.pt);
    S.abuf = reinterpret_cast<float*>(o + ao.abuf);
    S.sc = reinterpret_cast<float*>(o + ao.sc);
    S.cs = reinterpret_cast<float*>(o + ao.cs);
    S.kn = reinterpret_cast<bf16*>(o + ao.kn);
    S.vn = reinterpret_cast<bf16*>(o + ao.vn);
    S.mland = reinterpret_cast<float*>(o + ao.mland);
  }
  S.layers = reinterpret_cast<const DsLayer*>(sbase + lay.layers);
  int* s_sched = reinterpret_cast<int*>(sbase + lay.sched);
  S.off = s_sched;
  S.items = s_sched + DS_PHASES + 1;
  S.seq = s_seq;
  S.pos = s_pos;
  S.full = s_full;
  S.empty = s_empty;
  S.ids = s_ids;
  S.mrun = s_m;
  S.lrun = s_l;
  S.alpha = s_alpha;
  S.rs = s_rs;
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
  // the step's embedding rows into h_ll as layer -1's output, each CTA a slice (read by layer 0's QKV
  // staging and output projection)
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.T * p.H; i += gridDim.x * blockDim.x) {
    const int t = i / p.H;
    ll_store(p.h_ll + i, __bfloat162float(p.embed[packed_offset(s_ids[t], i - t * p.H, p.H)]), ds_tag(epoch, -1, DS_DOWN));
  }
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
