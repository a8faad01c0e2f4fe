// sample_filter.cu -- top-k / top-p filtered Gumbel-max sampling over float32 logits, one thread-block
// cluster of 2-8 CTAs per row.
//
// "19. Fast decode", section "Sampling without the CPU": the filters drop logits (to -inf) before the
// argmax, with shapes that do not depend on the data.  Definitions, with every integer decision exact:
//   * rank order: larger logit first, equal logits (+0 == -0) by increasing index; as one unsigned 64-bit
//     rank key per entry, (order-preserving bits of z) << 32 | ~v, larger key = earlier rank;
//   * top-k keeps the first k entries (k <= 0 or k >= V: off);
//   * top-p works on softmax(s), s = z * (1/T) in float32, over the top-k survivors: weight
//     w = floor(exp_rn(s - s_max) * 2^32) (integer), and an entry survives iff the weight of the survivors
//     ahead of it is <= (P * W - 1) >> 24 for W the total weight and P = p in units of 2^-24; that is the
//     shortest prefix whose mass reaches p, taken in integers so that no summation order matters;
//   * the draw is the unfiltered sampler's key s + g over the survivors, ties to the lowest index.
//
// The kernel finds each filter's boundary without sorting the vocabulary.  The row is spread over the
// cluster's CTAs; a histogram over kBuckets (2048) buckets of s_max - s (monotone in the rank order, so
// every bucket is a contiguous run of ranks) holds each bucket's count and integer weight, summed over the
// cluster in distributed shared memory; prefix sums over the buckets name the bucket holding the boundary.
// When every top-k candidate fits (kGatherCap entries) they are gathered and rank-sorted in shared memory;
// otherwise the boundary bucket alone is sorted (bitonic) or, when larger, resolved by a radix descent over
// the rank keys.  The Philox noise and the two logarithms run for survivors only.
#include <cooperative_groups.h>

#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace grd {

namespace cg = cooperative_groups;

namespace {

constexpr int kFThreads = 1024;
constexpr int kFWarps = kFThreads / 32;
constexpr int kBuckets = 2048;
constexpr int kGatherCap = kFilterGatherCap;
constexpr int kMaxCluster = 8;
constexpr unsigned kFull = 0xffffffffu;

// e^d for float32 d <= 0 from correctly rounded operations only (no contraction), 0 below -23:
// n = rint(d / ln 2), r = d - n ln2_hi - n ln2_lo (Cody and Waite), e^r by Taylor to r^7 / 7! in Horner
// form, times 2^n from the exponent bits (exact).  |n| <= 34, so n * ln2_hi (12 significant bits) is exact.
ENG_DEVICE float exp_rn(float d) {
  if (!(d >= -23.0f)) return 0.0f;
  const float inv_ln2 = __uint_as_float(0x3FB8AA3Bu);  // float32(1 / ln 2)
  const float ln2_hi = __uint_as_float(0x3F317000u);   // ln 2 with its low 12 mantissa bits cleared
  const float ln2_lo = __uint_as_float(0x3805FDF4u);   // float32(ln 2 - ln2_hi)
  const float n = rintf(__fmul_rn(d, inv_ln2));
  float r = __fsub_rn(d, __fmul_rn(n, ln2_hi));
  r = __fsub_rn(r, __fmul_rn(n, ln2_lo));
  float p = __uint_as_float(0x39500D01u);              // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3AB60B61u));  // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3C088889u));  // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3D2AAAABu));  // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(0x3E2AAAABu));  // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const float scale = __uint_as_float((uint32_t)((int)n + 127) << 23);
  return __fmul_rn(p, scale);
}

// Order-preserving unsigned image of a float, with -0 mapped onto +0.
ENG_DEVICE uint32_t ord_bits(float z) {
  uint32_t f = __float_as_uint(z);
  if (f == 0x80000000u) f = 0u;
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

ENG_DEVICE float from_ord(uint32_t o) { return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o); }

ENG_DEVICE unsigned long long rank_key(float z, uint32_t v) {
  return ((unsigned long long)ord_bits(z) << 32) | (unsigned long long)(~v);
}

ENG_DEVICE unsigned long long weight_of(float z, float inv_t, float s_max) {
  const float e = exp_rn(__fsub_rn(__fmul_rn(z, inv_t), s_max));
  return (unsigned long long)__float2ull_rz(__fmul_rn(e, 4294967296.0f));  // exact scaling, then floor
}

struct RowView {
  const float* z;
  int V;
  float inv_t, s_max, scale;
};

// Bucket of a finite logit: floor((s_max - s) * scale), clamped; non-decreasing along the rank order.
ENG_DEVICE int bucket_of(const RowView& rv, float z) {
  const float d = __fsub_rn(rv.s_max, __fmul_rn(z, rv.inv_t));
  const int b = __float2int_rz(__fmul_rn(d, rv.scale));
  return b < 0 ? 0 : (b >= kBuckets ? kBuckets - 1 : b);
}

ENG_DEVICE bool finite(float z) { return (__float_as_uint(z) & 0x7F800000u) != 0x7F800000u; }

// ------------------------------------------------------------------ one row over a cluster of C CTAs
//
// CTA c of the cluster streams the row slice [c * Vc, min(V, (c + 1) * Vc)), Vc a multiple of 4, with four
// 16-byte loads in flight per thread (the row stays in L2 between passes).  Every merge of the row's state
// is pushed into the other CTAs' shared memory (distributed shared memory) and followed by a cluster
// barrier, after which each CTA reads only its own copy; every decision is an integer computed identically
// in every CTA, so the CTAs never disagree.

struct Slice {
  const float* z;  // the whole row
  int lo, hi;      // this CTA's entries
  bool vec;        // the row starts on a 16-byte boundary
};

// visit calls f(v, x, valid) for every entry of the slice, 8 per thread per round, the next round's loads
// in flight while f runs.  Every thread of the CTA runs the same number of rounds and calls f 8 times per
// round (valid = false past the end), so f may hold warp-synchronous code.
template <int U>
ENG_DEVICE void load_round(const Slice& sl, int g0, float4 (&buf)[U]) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int v0 = sl.lo + 4 * (g0 + u * kFThreads + (int)threadIdx.x);
    if (sl.vec && v0 + 3 < sl.hi) {
      buf[u] = __ldg(reinterpret_cast<const float4*>(sl.z + v0));
    } else {
      buf[u].x = v0 < sl.hi ? __ldg(sl.z + v0) : 0.f;
      buf[u].y = v0 + 1 < sl.hi ? __ldg(sl.z + v0 + 1) : 0.f;
      buf[u].z = v0 + 2 < sl.hi ? __ldg(sl.z + v0 + 2) : 0.f;
      buf[u].w = v0 + 3 < sl.hi ? __ldg(sl.z + v0 + 3) : 0.f;
    }
  }
}

template <class F>
ENG_DEVICE void visit(const Slice& sl, F&& f) {
  constexpr int U = 2;
  const int groups = (sl.hi - sl.lo + 3) >> 2;
  if (groups <= 0) return;  // (uniform: the slice is the CTA's)
  float4 cur[U], nxt[U];
  load_round<U>(sl, 0, cur);
  for (int g0 = 0; g0 < groups; g0 += U * kFThreads) {
    if (g0 + U * kFThreads < groups) load_round<U>(sl, g0 + U * kFThreads, nxt);  // next round in flight
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v0 = sl.lo + 4 * (g0 + u * kFThreads + (int)threadIdx.x);
      f(v0, cur[u].x, v0 < sl.hi);
      f(v0 + 1, cur[u].y, v0 + 1 < sl.hi);
      f(v0 + 2, cur[u].z, v0 + 2 < sl.hi);
      f(v0 + 3, cur[u].w, v0 + 3 < sl.hi);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) cur[u] = nxt[u];
  }
}

ENG_DEVICE void cl_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
ENG_DEVICE void cl_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
ENG_DEVICE void cl_sync() {
  cl_arrive();
  cl_wait();
}

// ------------------------------------------------------------------ block reductions (1024 threads)
ENG_DEVICE unsigned long long warp_max_u64(unsigned long long x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(kFull, x, o);
    x = y > x ? y : x;
  }
  return x;
}

ENG_DEVICE unsigned long long warp_sum_u64(unsigned long long x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

template <bool MAX>
ENG_DEVICE unsigned long long block_reduce(unsigned long long x, unsigned long long* red) {
  x = MAX ? warp_max_u64(x) : warp_sum_u64(x);
  __syncthreads();  // red may still be read by a previous reduction
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  unsigned long long r = red[0];
  for (int w = 1; w < kFWarps; ++w) r = MAX ? (red[w] > r ? red[w] : r) : r + red[w];
  return r;
}

// Histogram add with warp aggregation when every member lane of the warp hits the same bin (runs of equal
// logits), per-lane shared atomics otherwise.  All 32 lanes must call it together.
template <bool MASS, bool KMAX>
ENG_DEVICE void hist_add(bool in, int bin, unsigned long long w, unsigned long long key, uint32_t* cnt,
                         unsigned long long* mass, unsigned long long* kmax) {
  const unsigned gm = __ballot_sync(kFull, in);
  if (!gm) return;
  const int leader = __ffs(gm) - 1;
  const int b0 = __shfl_sync(kFull, bin, leader);
  if (__all_sync(kFull, !in || bin == b0)) {
    const unsigned long long ws = MASS ? warp_sum_u64(in ? w : 0ull) : 0ull;
    const unsigned long long km = KMAX ? warp_max_u64(in ? key : 0ull) : 0ull;
    if ((int)(threadIdx.x & 31) == leader) {
      atomicAdd(&cnt[b0], (uint32_t)__popc(gm));
      if constexpr (MASS) atomicAdd(&mass[b0], ws);
      if constexpr (KMAX) atomicMax(&kmax[b0], km);
    }
  } else if (in) {
    atomicAdd(&cnt[bin], 1u);
    if constexpr (MASS) atomicAdd(&mass[bin], w);
    if constexpr (KMAX) atomicMax(&kmax[bin], key);
  }
}

// In-place inclusive prefix sums over kBuckets entries, kBuckets / kFThreads consecutive entries a thread.
template <typename T>
ENG_DEVICE void block_inclusive_scan(T* a, T* warp_tot) {
  constexpr int E = kBuckets / kFThreads;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  T v[E];
  T run = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    run += a[E * t + i];
    v[i] = run;
  }
  T incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  T base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  const T ex = base + incl - run;
#pragma unroll
  for (int i = 0; i < E; ++i) a[E * t + i] = ex + v[i];
  __syncthreads();
}

struct FShared {
  unsigned long long red[kFWarps];
  uint32_t cnt_tot[kFWarps];
  unsigned long long mass_tot[kFWarps];
  // pushed partials, [exchange][source CTA], each exchange used once: row max, row min, top-k weight inside
  // an oversized bucket, best draw, survivor count
  unsigned long long xchg[5][kMaxCluster];
  int gather_n;
  int sel_bin;
  unsigned long long sel_a, sel_b;
  // radix descent (large boundary buckets): this CTA's digit histogram
  uint32_t dcnt[256];
  unsigned long long dmass[256];
  unsigned long long dmax[256];
};

struct Row {
  cg::cluster_group cl;
  int C, me;
  Slice sl;
  RowView rv;
  FShared* sh;
  uint32_t* cnt;             // [kBuckets]
  unsigned long long* mass;  // [kBuckets]
  uint32_t* inc_cnt;         // [kBuckets] partial histograms pushed by the cluster, [source][bucket in range]
  unsigned long long* inc_mass;
  unsigned long long* keys;  // [kGatherCap]
};

template <class T>
ENG_DEVICE T* at_rank(const Row& w, T* p, int rank) {
  return w.cl.map_shared_rank(p, rank);
}

// Exact boundary inside one oversized bucket: radix descent over the rank keys of the group (entries of
// bucket gb with key >= kmin), 8 bits a level from the top, digit histograms summed over the cluster.
// COUNT mode returns the key at 0-based position `target`; otherwise the key of the last entry whose
// weight ahead, base + (group weight ahead of it), is <= thr.  Levels stop early when the chosen digit
// holds a single entry.  The digit histograms of the cluster land in the keys area.
template <bool COUNT>
ENG_DEVICE unsigned long long descend(Row& w, int gb, unsigned long long kmin, unsigned long long target,
                                      unsigned long long base, unsigned long long thr) {
  FShared& sh = *w.sh;
  uint32_t* in_cnt = reinterpret_cast<uint32_t*>(w.keys);                                  // [C][256]
  unsigned long long* in_mass = w.keys + kMaxCluster * 128;                                // [C][256]
  unsigned long long* in_max = w.keys + kMaxCluster * 128 + kMaxCluster * 256;             // [C][256]
  unsigned long long prefix = 0ull, ahead = COUNT ? 0ull : base;
  cl_sync();  // every CTA is done with its keys area before the first level lands there
  for (int level = 0; level < 8; ++level) {
    const int shift = 56 - 8 * level;
    for (int i = threadIdx.x; i < 256; i += kFThreads) {
      sh.dcnt[i] = 0u;
      sh.dmass[i] = 0ull;
      sh.dmax[i] = 0ull;
    }
    __syncthreads();
    visit(w.sl, [&](int v, float z, bool valid) {
      bool in = false;
      unsigned long long key = 0ull, wt = 0ull;
      if (valid && finite(z) && bucket_of(w.rv, z) == gb) {
        key = rank_key(z, (uint32_t)v);
        in = key >= kmin && (level == 0 || (key >> (shift + 8)) == prefix);
        if (in && !COUNT) wt = weight_of(z, w.rv.inv_t, w.rv.s_max);
      }
      hist_add<!COUNT, true>(in, (int)((key >> shift) & 255ull), wt, key, sh.dcnt, sh.dmass, sh.dmax);
    });
    __syncthreads();
    for (int i = threadIdx.x; i < 256 * w.C; i += kFThreads) {  // push to every CTA, slot [me][digit]
      const int t = i >> 8, d = i & 255;
      at_rank(w, in_cnt, t)[w.me * 256 + d] = sh.dcnt[d];
      at_rank(w, in_mass, t)[w.me * 256 + d] = sh.dmass[d];
      at_rank(w, in_max, t)[w.me * 256 + d] = sh.dmax[d];
    }
    cl_sync();
    if (threadIdx.x == 0) {
      int chosen = -1;
      unsigned long long chosen_ahead = ahead, chosen_cnt = 0ull, chosen_max = 0ull;
      for (int d = 255; d >= 0; --d) {
        unsigned long long c = 0ull, m = 0ull, mx = 0ull;
        for (int t = 0; t < w.C; ++t) {
          c += in_cnt[t * 256 + d];
          m += in_mass[t * 256 + d];
          mx = in_max[t * 256 + d] > mx ? in_max[t * 256 + d] : mx;
        }
        if (c == 0ull) continue;
        if (COUNT) {
          if (ahead + c > target) {
            chosen = d;
            chosen_ahead = ahead;
            chosen_cnt = c;
            chosen_max = mx;
            break;
          }
          ahead += c;
        } else {
          if (ahead > thr) break;  // the first entry of this digit is dropped, and so is everything after it
          chosen = d;
          chosen_ahead = ahead;
          chosen_cnt = c;
          chosen_max = mx;
          ahead += m;
        }
      }
      if (chosen < 0) chosen = 0;  // unreachable for a non-empty group with a reachable target
      sh.sel_bin = chosen;
      sh.sel_a = chosen_ahead;
      sh.sel_b = chosen_cnt == 1ull ? chosen_max : 0ull;
    }
    __syncthreads();
    const int d = sh.sel_bin;
    ahead = sh.sel_a;
    prefix = (prefix << 8) | (unsigned long long)d;
    const unsigned long long single = sh.sel_b;
    cl_sync();  // every CTA has read this level's histograms before the next level overwrites them
    if (single) return single;
  }
  return prefix;
}

// Gather the rank keys of buckets [b_lo, b_hi] from the whole cluster into every CTA's keys[0, n) and sort
// them in decreasing order (bitonic over the next power of two, padded with 0, which is below every real
// key).  Each warp reserves room for its matches with one remote atomic per CTA.  Returns n (<= kGatherCap;
// the caller checks the buckets' count first).
ENG_DEVICE int gather_sorted(Row& w, int b_lo, int b_hi) {
  FShared& sh = *w.sh;
  if (threadIdx.x == 0) sh.gather_n = 0;
  cl_sync();  // counters cleared, and every CTA is done with its previous keys
  const unsigned lane = threadIdx.x & 31;
  visit(w.sl, [&](int v, float z, bool valid) {
    bool match = false;
    if (valid && finite(z)) {
      const int b = bucket_of(w.rv, z);
      match = b >= b_lo && b <= b_hi;
    }
    const unsigned m = __ballot_sync(kFull, match);
    if (!m) return;
    const int here = __popc(m & ((1u << lane) - 1u));
    int base = 0;
    if ((int)lane < w.C) base = atomicAdd(at_rank(w, &sh.gather_n, (int)lane), __popc(m));
    const unsigned long long key = rank_key(z, (uint32_t)v);
    for (int t = 0; t < w.C; ++t) {
      const int slot = __shfl_sync(kFull, base, t) + here;
      if (match && slot < kGatherCap) at_rank(w, w.keys, t)[slot] = key;
    }
  });
  cl_sync();
  unsigned long long* keys = w.keys;
  const int n = sh.gather_n < kGatherCap ? sh.gather_n : kGatherCap;
  if (n <= kFThreads) {  // rank sort: the keys are distinct, so entry t goes to #(larger keys)
    unsigned long long* out = w.inc_mass;  // free once the histograms are merged
    if ((int)threadIdx.x < n) {
      const unsigned long long my = keys[threadIdx.x];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += keys[j] > my;
      out[rank] = my;
    }
    __syncthreads();
    if ((int)threadIdx.x < n) keys[threadIdx.x] = out[threadIdx.x];
    __syncthreads();
    return n;
  }
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  for (int i = n + threadIdx.x; i < n2; i += kFThreads) keys[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (n2 >> 1); i += kFThreads) {
        const int lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
        const bool first_half = (lo & size) == 0;  // this run ends up decreasing
        const unsigned long long a = keys[lo], b = keys[hi];
        if (first_half ? (a < b) : (a > b)) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  return n;
}

// Sum of the top-p weights of keys[0, n) (sorted keys of this CTA).
ENG_DEVICE unsigned long long sorted_weight(Row& w, int n) {
  unsigned long long part = 0ull;
  for (int i = threadIdx.x; i < n; i += kFThreads)
    part += weight_of(from_ord((uint32_t)(w.keys[i] >> 32)), w.rv.inv_t, w.rv.s_max);
  return block_reduce<false>(part, w.sh->red);
}

// Top-p survivors among the sorted keys[0, lim) whose first entry has weight A ahead of it: the length of
// the prefix whose weight ahead (A + exclusive prefix sum in rank order) is <= thr; at least 1.
ENG_DEVICE int prefix_cut(Row& w, int lim, unsigned long long A, unsigned long long thr) {
  FShared& sh = *w.sh;
  __syncthreads();  // the caller may still be reading sel_bin
  if (threadIdx.x == 0) {
    sh.sel_a = A;    // running weight ahead of the current round
    sh.sel_bin = 1;  // survivors so far (the first entry always survives)
  }
  __syncthreads();
  for (int c0 = 0; c0 < lim; c0 += kFThreads) {
    const int i = c0 + threadIdx.x;
    const unsigned long long wt =
        i < lim ? weight_of(from_ord((uint32_t)(w.keys[i] >> 32)), w.rv.inv_t, w.rv.s_max) : 0ull;
    unsigned long long incl = wt;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.mass_tot[warp] = incl;
    __syncthreads();
    unsigned long long before = sh.sel_a;
    for (int ww = 0; ww < warp; ++ww) before += sh.mass_tot[ww];
    const unsigned long long ahead = before + incl - wt;
    if (i < lim && ahead <= thr) atomicMax(&sh.sel_bin, i + 1);
    __syncthreads();
    if (threadIdx.x == kFThreads - 1) sh.sel_a = ahead + wt;
    __syncthreads();
  }
  return sh.sel_bin;
}

// Whether every candidate of top-k (the buckets up to the one holding rank k - 1) fits in shared memory;
// cnt holds inclusive prefix counts, so that bucket's inclusive count is the smallest one >= k.
ENG_DEVICE bool top_k_fits(const uint32_t* cnt, int top_k) {
  int lo = 0, hi = kBuckets - 1;  // first bucket with cnt >= k (cnt is non-decreasing)
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cnt[mid] >= (uint32_t)top_k) hi = mid;
    else lo = mid + 1;
  }
  return cnt[lo] <= (uint32_t)kGatherCap;
}

// The cut's bound: weight ahead <= (P * W - 1) >> 24, i.e. (weight ahead) * 2^24 < P * W.
ENG_DEVICE unsigned long long top_p_bound(unsigned long long P, unsigned long long W) {
  const unsigned __int128 pw = (unsigned __int128)P * (unsigned __int128)W;
  return (unsigned long long)((pw - 1u) >> 24);
}

}  // namespace

__global__ void __launch_bounds__(kFThreads, 1) k_sample_filtered(FilterParams p) {
  extern __shared__ __align__(16) uint8_t f_smem[];
  __shared__ FShared sh;
  Row w{cg::this_cluster()};
  w.C = (int)w.cl.num_blocks();
  w.me = (int)w.cl.block_rank();
  w.sh = &sh;
  w.cnt = reinterpret_cast<uint32_t*>(f_smem);
  w.inc_cnt = w.cnt + kBuckets;
  w.mass = reinterpret_cast<unsigned long long*>(f_smem + kBuckets * 8);
  w.inc_mass = w.mass + kBuckets;
  w.keys = reinterpret_cast<unsigned long long*>(f_smem + kBuckets * 24);

  const int r = blockIdx.y, V = p.vocab;
  const float* z = p.logits + (size_t)r * V;
  const float it = p.inv_temp[r];
  const int top_k = p.top_k ? p.top_k[r] : 0;
  const unsigned long long P = p.p_units ? (unsigned long long)(uint32_t)p.p_units[r] : 0ull;
  bool kon = top_k > 0 && top_k < V;
  const bool pon = P > 0ull && P < (1ull << 24);
  if (p.only_filtered && (it == 0.0f || (!kon && !pon))) {  // the caller's draw stands (whole cluster)
    if (p.row_ext && w.me == 0 && threadIdx.x == 0) {
      p.row_ext[2 * r] = 0u;
      p.row_ext[2 * r + 1] = 0u;
    }
    return;
  }
  // extremes formed by the producer of the logits (sampled rows only: greedy rows need the argmax index)
  const bool given_ext = p.row_ext && it != 0.0f;
  uint32_t ext_max = 0u, ext_min_inv = 0u;
  if (given_ext) {
    ext_max = p.row_ext[2 * r];
    ext_min_inv = p.row_ext[2 * r + 1];
  }
  cl_arrive();  // every CTA has started (and read the extremes) before any write into shared memory
  const uint32_t rng[4] = {p.rng[0], p.rng[1], p.rng[2], p.rng[3]};
  const float* keys = (p.keys && *p.keys_valid) ? p.keys : nullptr;
  const int Vc = (((V + w.C - 1) / w.C) + 3) & ~3;
  w.sl.z = z;
  w.sl.lo = w.me * Vc < V ? w.me * Vc : V;
  w.sl.hi = w.sl.lo + Vc < V ? w.sl.lo + Vc : V;
  w.sl.vec = (reinterpret_cast<uintptr_t>(z) & 15) == 0;

  // extremes of the finite logits of the row (order-preserving bits; with the index for greedy rows),
  // flagging non-finite ones
  unsigned long long kmax = 0ull, kmin_inv = 0ull;
  if (given_ext) {
    kmax = (unsigned long long)ext_max << 32;
    kmin_inv = (unsigned long long)ext_min_inv << 32;
    cl_wait();
  } else {
    bool bad = false;
    if (it == 0.0f) {
      visit(w.sl, [&](int v, float x, bool valid) {
        if (!valid) return;
        if (!finite(x)) {
          bad = true;
          return;
        }
        const unsigned long long k = rank_key(x, (uint32_t)v);
        kmax = k > kmax ? k : kmax;
      });
    } else {
      uint32_t omax = 0u, omin_inv = 0u;
      visit(w.sl, [&](int v, float x, bool valid) {
        if (!valid) return;
        if (!finite(x)) {
          bad = true;
          return;
        }
        const uint32_t o = ord_bits(x);
        omax = o > omax ? o : omax;
        omin_inv = ~o > omin_inv ? ~o : omin_inv;
      });
      kmax = (unsigned long long)omax << 32;
      kmin_inv = (unsigned long long)omin_inv << 32;
    }
    if (bad) set_status(p.status, ST_NAN);
    kmax = block_reduce<true>(kmax, sh.red);
    kmin_inv = block_reduce<true>(kmin_inv, sh.red);
    cl_wait();
    if (threadIdx.x < (unsigned)w.C) {
      at_rank(w, &sh.xchg[0][0], threadIdx.x)[w.me] = kmax;
      at_rank(w, &sh.xchg[1][0], threadIdx.x)[w.me] = kmin_inv;
    }
    cl_sync();
    for (int t = 0; t < w.C; ++t) {
      kmax = sh.xchg[0][t] > kmax ? sh.xchg[0][t] : kmax;
      kmin_inv = sh.xchg[1][t] > kmin_inv ? sh.xchg[1][t] : kmin_inv;
    }
  }
  if (p.row_ext && w.me == 0 && threadIdx.x == 0) {  // every CTA has read them: ready for the next step
    p.row_ext[2 * r] = 0u;
    p.row_ext[2 * r + 1] = 0u;
  }
  if (kmax == 0ull || it == 0.0f) {  // no finite logit / greedy: neither filter can drop the top entry
    if (w.me == 0 && threadIdx.x == 0) {
      p.out_ids[r] = kmax ? (int)(~(uint32_t)(kmax & 0xFFFFFFFFull)) : 0;
      if (p.out_kept) p.out_kept[r] = kmax ? 1 : 0;
    }
    return;  // nothing reads this CTA's shared memory any more
  }
  const float zmax = from_ord((uint32_t)(kmax >> 32)), zmin = from_ord((uint32_t)((~kmin_inv) >> 32));
  w.rv.z = z;
  w.rv.V = V;
  w.rv.inv_t = it;
  w.rv.s_max = __fmul_rn(zmax, it);
  const float range = __fsub_rn(w.rv.s_max, __fmul_rn(zmin, it));
  float scale = range > 0.0f ? __fdiv_rn((float)kBuckets, range) : 0.0f;
  if (!(scale < 3.0e38f)) scale = 0.0f;
  w.rv.scale = scale;

  unsigned long long threshold = 0ull;  // survivors: rank key >= threshold
  unsigned long long best = 0ull, kept = 0ull;
  bool drawn = false;  // the draw already ran over a sorted candidate list
  if (kon || pon) {  // (uniform across the cluster: every branch below holds barriers)
    uint32_t* cnt = w.cnt;
    unsigned long long* mass = w.mass;
    // The weights are needed per bucket only when the candidates may not all fit in shared memory.
    bool have_mass = pon && (!kon || top_k > kGatherCap);
    for (int pass = 0; pass < 2; ++pass) {
      for (int i = threadIdx.x; i < kBuckets; i += kFThreads) {
        cnt[i] = 0u;
        mass[i] = 0ull;
      }
      __syncthreads();
      visit(w.sl, [&](int v, float x, bool valid) {
        const bool in = valid && finite(x);
        const int b = in ? bucket_of(w.rv, x) : 0;
        if (have_mass) {
          const unsigned long long wt = in ? weight_of(x, it, w.rv.s_max) : 0ull;
          hist_add<true, false>(in, b, wt, 0ull, cnt, mass, nullptr);
        } else {
          hist_add<false, false>(in, b, 0ull, 0ull, cnt, nullptr, nullptr);
        }
      });
      __syncthreads();
      // cluster sum: bucket i belongs to CTA i / Rg, which receives every CTA's partial at [source][i % Rg],
      // sums them and writes the total into every CTA's histogram
      // (a second pass is safe: every CTA has passed the first pass's last barrier, after its reads)
      const int Rg = kBuckets / w.C;
      for (int i = threadIdx.x; i < kBuckets; i += kFThreads) {
        const int o = i / Rg, j = i - o * Rg;
        at_rank(w, w.inc_cnt, o)[w.me * Rg + j] = cnt[i];
        if (have_mass) at_rank(w, w.inc_mass, o)[w.me * Rg + j] = mass[i];
      }
      cl_sync();
      for (int j = threadIdx.x; j < Rg; j += kFThreads) {
        uint32_t c = 0u;
        unsigned long long m = 0ull;
        for (int t = 0; t < w.C; ++t) {
          c += w.inc_cnt[t * Rg + j];
          if (have_mass) m += w.inc_mass[t * Rg + j];
        }
        for (int t = 0; t < w.C; ++t) {
          at_rank(w, cnt, t)[w.me * Rg + j] = c;
          if (have_mass) at_rank(w, mass, t)[w.me * Rg + j] = m;
        }
      }
      cl_sync();
      block_inclusive_scan<uint32_t>(cnt, sh.cnt_tot);
      if (have_mass) block_inclusive_scan<unsigned long long>(mass, sh.mass_tot);
      if (kon && (uint32_t)top_k >= cnt[kBuckets - 1]) kon = false;  // k covers every finite logit
      if (!pon || have_mass || (kon && cnt[kBuckets - 1] > 0u && top_k_fits(cnt, top_k))) break;
      have_mass = true;  // the candidates overflow shared memory: count the weights too
    }

    // ---- top-k: bucket bk holds rank k - 1
    int bk = kBuckets - 1, sorted_bucket = -1, sorted_n = 0;
    unsigned long long key_k = 0ull, kept_mass_bk = 0ull;
    uint32_t kept_in_bk = 0u;
    if (kon) {
      const uint32_t want = (uint32_t)top_k - 1u;
      if (threadIdx.x == 0) sh.sel_bin = kBuckets - 1;
      __syncthreads();
      for (int b = threadIdx.x; b < kBuckets; b += kFThreads) {
        const uint32_t ex = b ? cnt[b - 1] : 0u;
        if (ex <= want && want < cnt[b]) sh.sel_bin = b;
      }
      __syncthreads();
      bk = sh.sel_bin;
      if (cnt[bk] <= (uint32_t)kGatherCap) {
        // every candidate (buckets 0..bk) sorted in shared memory: top-k, the top-p cut and the draw
        gather_sorted(w, 0, bk);
        int n_keep = top_k;
        if (pon) {
          const unsigned long long W = sorted_weight(w, top_k);
          n_keep = prefix_cut(w, top_k, 0ull, top_p_bound(P, W));
        }
        for (int i = w.me * kFThreads + threadIdx.x; i < n_keep; i += w.C * kFThreads) {
          const unsigned long long k = w.keys[i];
          const uint32_t v = ~(uint32_t)(k & 0xFFFFFFFFull);
          const float key = keys ? keys[(size_t)r * V + v]
                                   : sample_key(from_ord((uint32_t)(k >> 32)), it, rng, (uint32_t)r, v);
          const unsigned long long pk = pack_key_index(key, v);
          best = pk > best ? pk : best;
        }
        kept = (w.me == 0 && threadIdx.x == 0) ? (unsigned long long)n_keep : 0ull;  // summed over the cluster
        drawn = true;
      } else {
        const uint32_t ex = bk ? cnt[bk - 1] : 0u, nb = cnt[bk] - ex;
        const uint32_t j = want - ex;  // position inside the bucket
        kept_in_bk = j + 1u;
        if (nb <= (uint32_t)kGatherCap) {
          sorted_n = gather_sorted(w, bk, bk);
          sorted_bucket = bk;
          key_k = w.keys[j];
          if (pon) kept_mass_bk = sorted_weight(w, (int)kept_in_bk);
        } else {
          key_k = descend<true>(w, bk, 0ull, j, 0ull, 0ull);
          if (pon) {
            unsigned long long part = 0ull;
            visit(w.sl, [&](int v, float x, bool valid) {
              if (valid && finite(x) && bucket_of(w.rv, x) == bk && rank_key(x, (uint32_t)v) >= key_k)
                part += weight_of(x, it, w.rv.s_max);
            });
            part = block_reduce<false>(part, sh.red);
            if (threadIdx.x < (unsigned)w.C) at_rank(w, &sh.xchg[2][0], threadIdx.x)[w.me] = part;
            cl_sync();
            kept_mass_bk = 0ull;
            for (int t = 0; t < w.C; ++t) kept_mass_bk += sh.xchg[2][t];
          }
        }
        threshold = key_k;
      }
    }

    // ---- top-p over the top-k survivors (candidates too many for shared memory)
    if (pon && !drawn) {
      const unsigned long long W = kon ? ((bk ? mass[bk - 1] : 0ull) + kept_mass_bk) : mass[kBuckets - 1];
      const unsigned long long thr = top_p_bound(P, W);
      // last non-empty eligible bucket whose first entry survives (weight ahead of it <= thr)
      const int blim = kon ? bk : kBuckets - 1;
      if (threadIdx.x == 0) sh.sel_bin = 0;
      __syncthreads();
      for (int b = threadIdx.x; b <= blim; b += kFThreads) {
        const unsigned long long ex = b ? mass[b - 1] : 0ull;
        const uint32_t nb = cnt[b] - (b ? cnt[b - 1] : 0u);
        if (nb > 0u && ex <= thr) atomicMax(&sh.sel_bin, b);
      }
      __syncthreads();
      const int bp = sh.sel_bin;
      const unsigned long long A = bp ? mass[bp - 1] : 0ull;
      const uint32_t nbp = cnt[bp] - (bp ? cnt[bp - 1] : 0u);
      const unsigned long long kfloor = (kon && bp == bk) ? key_k : 0ull;
      if (nbp <= (uint32_t)kGatherCap) {
        if (sorted_bucket != bp) sorted_n = gather_sorted(w, bp, bp);
        const int lim = (kon && bp == bk) ? (int)kept_in_bk : sorted_n;
        threshold = w.keys[prefix_cut(w, lim, A, thr) - 1];
        __syncthreads();
      } else {
        threshold = descend<false>(w, bp, kfloor, 0ull, A, thr);
      }
    }
  }

  // ---- the draw over the survivors of the slice, then over the cluster (pushed to CTA 0)
  if (!drawn) {
    visit(w.sl, [&](int v, float x, bool valid) {
      if (!valid || !finite(x) || rank_key(x, (uint32_t)v) < threshold) return;
      ++kept;
      const float key = keys ? keys[(size_t)r * V + v] : sample_key(x, it, rng, (uint32_t)r, (uint32_t)v);
      const unsigned long long pk = pack_key_index(key, (uint32_t)v);
      best = pk > best ? pk : best;
    });
  }
  best = block_reduce<true>(best, sh.red);
  kept = block_reduce<false>(kept, sh.red);
  if (threadIdx.x == 0) {
    at_rank(w, &sh.xchg[3][0], 0)[w.me] = best;
    at_rank(w, &sh.xchg[4][0], 0)[w.me] = kept;
  }
  cl_sync();  // after this, only CTA 0 reads, and only its own shared memory
  if (w.me == 0 && threadIdx.x == 0) {
    best = 0ull;
    kept = 0ull;
    for (int t = 0; t < w.C; ++t) {
      best = sh.xchg[3][t] > best ? sh.xchg[3][t] : best;
      kept += sh.xchg[4][t];
    }
    p.out_ids[r] = (int)unpack_index(best);
    if (p.out_kept) p.out_kept[r] = (int)kept;
  }
}

constexpr size_t kFilterSmem = (size_t)kBuckets * 24 + (size_t)kGatherCap * 8;

// Cluster size for `rows` rows: enough CTAs per row to cover the device's SMs, at most kMaxCluster.
static int filter_cluster(int rows) {
  const int sms = device_sm_count();
  int C = 1;
  while (C < kMaxCluster && rows * C * 2 <= sms) C <<= 1;
  return C;
}

cudaError_t launch_sample_filtered(const FilterParams& p, int rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(k_sample_filtered), (int)kFilterSmem);
  if (e != cudaSuccess) return e;
  const int C = filter_cluster(rows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, rows, 1);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = kFilterSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_sample_filtered, p);
}

__global__ void k_exp_rn(const float* d, float* out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = exp_rn(d[i]);
}

cudaError_t launch_exp_rn(const float* d, float* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8192) blocks = 8192;
  k_exp_rn<<<(unsigned)blocks, 256, 0, s>>>(d, out, n);
  return cudaGetLastError();
}

}  // namespace grd
