// sample_filter.cu -- top-k / top-p filtered Gumbel-max sampling over float32 logits, one CTA per row.
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
// The kernel finds each filter's boundary without sorting the vocabulary.  A histogram over 4096 buckets
// of s_max - s (monotone in the rank order, so every bucket is a contiguous run of ranks) holds each
// bucket's count and integer weight; prefix sums over the buckets name the bucket holding the boundary;
// that bucket alone is sorted in shared memory (bitonic, up to 8192 entries) or, when larger, resolved by a
// radix descent over the rank keys.  The Philox noise and the two logarithms run for survivors only.
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace grd {

namespace {

constexpr int kFThreads = 1024;
constexpr int kFWarps = kFThreads / 32;
constexpr int kBuckets = 4096;
constexpr int kGatherCap = 8192;
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

// ------------------------------------------------------------------ block reductions (1024 threads)
struct Red {
  unsigned long long u[kFWarps];
};

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
ENG_DEVICE unsigned long long block_reduce(unsigned long long x, Red& red) {
  x = MAX ? warp_max_u64(x) : warp_sum_u64(x);
  __syncthreads();  // red may still be read by a previous reduction
  if ((threadIdx.x & 31) == 0) red.u[threadIdx.x >> 5] = x;
  __syncthreads();
  unsigned long long r = red.u[0];
  for (int w = 1; w < kFWarps; ++w) r = MAX ? (red.u[w] > r ? red.u[w] : r) : r + red.u[w];
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

// In-place inclusive prefix sums over kBuckets entries, 4 consecutive entries per thread.
template <typename T>
ENG_DEVICE void block_inclusive_scan(T* a, T* warp_tot) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  T v0 = a[4 * t], v1 = v0 + a[4 * t + 1], v2 = v1 + a[4 * t + 2], v3 = v2 + a[4 * t + 3];
  T incl = v3;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  T base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  const T ex = base + incl - v3;
  a[4 * t] = ex + v0;
  a[4 * t + 1] = ex + v1;
  a[4 * t + 2] = ex + v2;
  a[4 * t + 3] = ex + v3;
  __syncthreads();
}

struct FShared {
  Red red;
  uint32_t cnt_tot[kFWarps];
  unsigned long long mass_tot[kFWarps];
  int gather_n;
  int sel_bin;
  unsigned long long sel_a, sel_b;
  // radix descent (large boundary buckets)
  uint32_t dcnt[256];
  unsigned long long dmass[256];
  unsigned long long dmax[256];
};

// Exact boundary inside one oversized bucket: radix descent over the rank keys of the group (entries of
// bucket gb with key >= kmin), 8 bits a level from the top.  COUNT mode returns the key at 0-based
// position `target`; otherwise the key of the last entry whose weight ahead, base + (group weight ahead of
// it), is <= thr.  Levels stop early when the chosen digit holds a single entry.
template <bool COUNT>
ENG_DEVICE unsigned long long descend(const RowView& rv, int gb, unsigned long long kmin, unsigned long long target,
                                      unsigned long long base, unsigned long long thr, FShared& sh) {
  unsigned long long prefix = 0ull, ahead = COUNT ? 0ull : base;
  for (int level = 0; level < 8; ++level) {
    const int shift = 56 - 8 * level;
    for (int i = threadIdx.x; i < 256; i += kFThreads) {
      sh.dcnt[i] = 0u;
      sh.dmass[i] = 0ull;
      sh.dmax[i] = 0ull;
    }
    __syncthreads();
    for (int base_v = 0; base_v < rv.V; base_v += kFThreads) {
      const int v = base_v + threadIdx.x;
      bool in = false;
      unsigned long long key = 0ull, w = 0ull;
      if (v < rv.V) {
        const float z = rv.z[v];
        if (finite(z) && bucket_of(rv, z) == gb) {
          key = rank_key(z, (uint32_t)v);
          in = key >= kmin && (level == 0 || (key >> (shift + 8)) == prefix);
          if (in && !COUNT) w = weight_of(z, rv.inv_t, rv.s_max);
        }
      }
      hist_add<!COUNT, true>(in, (int)((key >> shift) & 255ull), w, key, sh.dcnt, sh.dmass, sh.dmax);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int chosen = -1;
      unsigned long long chosen_ahead = ahead;
      for (int d = 255; d >= 0; --d) {
        if (sh.dcnt[d] == 0u) continue;
        if (COUNT) {
          if (ahead + sh.dcnt[d] > target) {
            chosen = d;
            chosen_ahead = ahead;
            break;
          }
          ahead += sh.dcnt[d];
        } else {
          if (ahead > thr) break;  // the first entry of this digit is dropped, and so is everything after it
          chosen = d;
          chosen_ahead = ahead;
          ahead += sh.dmass[d];
        }
      }
      if (chosen < 0) chosen = 0;  // unreachable for a non-empty group with a reachable target
      sh.sel_bin = chosen;
      sh.sel_a = chosen_ahead;
      sh.sel_b = sh.dcnt[chosen] == 1u ? sh.dmax[chosen] : 0ull;
    }
    __syncthreads();
    const int d = sh.sel_bin;
    ahead = sh.sel_a;
    prefix = (prefix << 8) | (unsigned long long)d;
    const unsigned long long single = sh.sel_b;
    __syncthreads();
    if (single) return single;
  }
  return prefix;
}

// Gather the rank keys of bucket gb into keys[0, n) and sort them in decreasing order (bitonic over the
// next power of two, padded with 0, which is below every real key).  Returns n.
ENG_DEVICE int gather_sorted(const RowView& rv, int gb, unsigned long long* keys, FShared& sh) {
  if (threadIdx.x == 0) sh.gather_n = 0;
  __syncthreads();
  for (int v = threadIdx.x; v < rv.V; v += kFThreads) {
    const float z = rv.z[v];
    if (finite(z) && bucket_of(rv, z) == gb) {
      const int slot = atomicAdd(&sh.gather_n, 1);
      if (slot < kGatherCap) keys[slot] = rank_key(z, (uint32_t)v);
    }
  }
  __syncthreads();
  const int n = sh.gather_n < kGatherCap ? sh.gather_n : kGatherCap;
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

}  // namespace

__global__ void __launch_bounds__(kFThreads, 1) k_sample_filtered(FilterParams p) {
  extern __shared__ __align__(16) uint8_t f_smem[];
  uint32_t* cnt = reinterpret_cast<uint32_t*>(f_smem);                                      // [kBuckets]
  unsigned long long* mass = reinterpret_cast<unsigned long long*>(f_smem + kBuckets * 4);   // [kBuckets]
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(f_smem + kBuckets * 12);  // [kGatherCap]
  __shared__ FShared sh;

  const int r = blockIdx.x, V = p.vocab;
  const float* z = p.logits + (size_t)r * V;
  const float it = p.inv_temp[r];
  const int top_k = p.top_k ? p.top_k[r] : 0;
  const unsigned long long P = p.p_units ? (unsigned long long)(uint32_t)p.p_units[r] : 0ull;
  bool kon = top_k > 0 && top_k < V;
  const bool pon = P > 0ull && P < (1ull << 24);
  if (p.only_filtered && (it == 0.0f || (!kon && !pon))) return;  // the caller's draw stands
  const uint32_t rng[4] = {p.rng[0], p.rng[1], p.rng[2], p.rng[3]};

  // extremes of the finite logits (and the greedy argmax), flagging non-finite ones
  unsigned long long kmax = 0ull, kmin_inv = 0ull;
  bool bad = false;
  for (int v = threadIdx.x; v < V; v += kFThreads) {
    const float x = z[v];
    if (!finite(x)) {
      bad = true;
      continue;
    }
    const unsigned long long k = rank_key(x, (uint32_t)v);
    kmax = k > kmax ? k : kmax;
    const unsigned long long ki = ~k;
    kmin_inv = ki > kmin_inv ? ki : kmin_inv;
  }
  if (bad) set_status(p.status, ST_NAN);
  kmax = block_reduce<true>(kmax, sh.red);
  kmin_inv = block_reduce<true>(kmin_inv, sh.red);
  if (kmax == 0ull) {  // no finite logit
    if (threadIdx.x == 0) {
      p.out_ids[r] = 0;
      if (p.out_kept) p.out_kept[r] = 0;
    }
    return;
  }
  if (it == 0.0f) {  // greedy: neither filter can drop the top entry
    if (threadIdx.x == 0) {
      p.out_ids[r] = (int)(~(uint32_t)(kmax & 0xFFFFFFFFull));
      if (p.out_kept) p.out_kept[r] = 1;
    }
    return;
  }
  const float zmax = from_ord((uint32_t)(kmax >> 32)), zmin = from_ord((uint32_t)((~kmin_inv) >> 32));
  RowView rv;
  rv.z = z;
  rv.V = V;
  rv.inv_t = it;
  rv.s_max = __fmul_rn(zmax, it);
  const float range = __fsub_rn(rv.s_max, __fmul_rn(zmin, it));
  float scale = range > 0.0f ? __fdiv_rn((float)kBuckets, range) : 0.0f;
  if (!(scale < 3.0e38f)) scale = 0.0f;
  rv.scale = scale;

  unsigned long long threshold = 0ull;  // survivors: rank key >= threshold
  if (kon || pon) {  // (uniform across the CTA: every branch below holds block-wide barriers)
    for (int i = threadIdx.x; i < kBuckets; i += kFThreads) {
      cnt[i] = 0u;
      mass[i] = 0ull;
    }
    __syncthreads();
    for (int base_v = 0; base_v < V; base_v += kFThreads) {
      const int v = base_v + threadIdx.x;
      bool in = false;
      int b = 0;
      unsigned long long w = 0ull;
      if (v < V) {
        const float x = z[v];
        if (finite(x)) {
          in = true;
          b = bucket_of(rv, x);
          if (pon) w = weight_of(x, it, rv.s_max);
        }
      }
      if (pon)
        hist_add<true, false>(in, b, w, 0ull, cnt, mass, nullptr);
      else
        hist_add<false, false>(in, b, 0ull, 0ull, cnt, nullptr, nullptr);
    }
    __syncthreads();
    block_inclusive_scan<uint32_t>(cnt, sh.cnt_tot);
    if (pon) block_inclusive_scan<unsigned long long>(mass, sh.mass_tot);
    if (kon && (uint32_t)top_k >= cnt[kBuckets - 1]) kon = false;  // k covers every finite logit

    // ---- top-k: bucket bk holds rank k - 1; its exact key by sorting that bucket
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
      const uint32_t ex = bk ? cnt[bk - 1] : 0u, nb = cnt[bk] - ex;
      const uint32_t j = want - ex;  // position inside the bucket
      kept_in_bk = j + 1u;
      if (nb <= (uint32_t)kGatherCap) {
        sorted_n = gather_sorted(rv, bk, keys, sh);
        sorted_bucket = bk;
        key_k = keys[j];
        if (pon) {
          unsigned long long part = 0ull;
          for (uint32_t i = threadIdx.x; i <= j; i += kFThreads) {
            const unsigned long long k = keys[i];
            part += weight_of(from_ord((uint32_t)(k >> 32)), it, rv.s_max);
          }
          kept_mass_bk = block_reduce<false>(part, sh.red);
        }
      } else {
        key_k = descend<true>(rv, bk, 0ull, j, 0ull, 0ull, sh);
        if (pon) {
          unsigned long long part = 0ull;
          for (int v = threadIdx.x; v < V; v += kFThreads) {
            const float x = z[v];
            if (finite(x) && bucket_of(rv, x) == bk && rank_key(x, (uint32_t)v) >= key_k)
              part += weight_of(x, it, rv.s_max);
          }
          kept_mass_bk = block_reduce<false>(part, sh.red);
        }
      }
      threshold = key_k;
    }

    // ---- top-p over the top-k survivors
    if (pon) {
      const unsigned long long W = kon ? ((bk ? mass[bk - 1] : 0ull) + kept_mass_bk) : mass[kBuckets - 1];
      const unsigned __int128 pw = (unsigned __int128)P * (unsigned __int128)W;
      const unsigned long long thr = (unsigned long long)((pw - 1u) >> 24);
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
        if (sorted_bucket != bp) sorted_n = gather_sorted(rv, bp, keys, sh);
        const int lim = (kon && bp == bk) ? (int)kept_in_bk : sorted_n;
        // weight ahead of each sorted entry: exclusive prefix sums in rank order, one pass per 1024 entries
        if (threadIdx.x == 0) sh.sel_a = A;  // running weight ahead of the current chunk
        if (threadIdx.x == 0) sh.gather_n = 1;  // survivors in this bucket (the first always survives)
        __syncthreads();
        for (int c0 = 0; c0 < lim; c0 += kFThreads) {
          const int i = c0 + threadIdx.x;
          const unsigned long long w = i < lim ? weight_of(from_ord((uint32_t)(keys[i] >> 32)), it, rv.s_max) : 0ull;
          // inclusive warp scan, then across warps
          unsigned long long incl = w;
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
          const unsigned long long ahead = before + incl - w;
          if (i < lim && ahead <= thr) atomicMax(&sh.gather_n, i + 1);
          __syncthreads();
          if (threadIdx.x == kFThreads - 1) sh.sel_a = ahead + w;
          __syncthreads();
        }
        threshold = keys[sh.gather_n - 1];
        __syncthreads();
      } else {
        threshold = descend<false>(rv, bp, kfloor, 0ull, A, thr, sh);
      }
    }
  }

  // ---- the draw over the survivors
  unsigned long long best = 0ull, kept = 0ull;
  for (int v = threadIdx.x; v < V; v += kFThreads) {
    const float x = z[v];
    if (!finite(x) || rank_key(x, (uint32_t)v) < threshold) continue;
    ++kept;
    const float key = sample_key(x, it, rng, (uint32_t)r, (uint32_t)v);
    const unsigned long long pk = pack_key_index(key, (uint32_t)v);
    best = pk > best ? pk : best;
  }
  best = block_reduce<true>(best, sh.red);
  kept = block_reduce<false>(kept, sh.red);
  if (threadIdx.x == 0) {
    p.out_ids[r] = (int)unpack_index(best);
    if (p.out_kept) p.out_kept[r] = (int)kept;
  }
}

constexpr size_t kFilterSmem = (size_t)kBuckets * 12 + (size_t)kGatherCap * 8;

cudaError_t launch_sample_filtered(const FilterParams& p, int rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  static bool attr_set = false;  // the attribute is per function, set once per process
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(k_sample_filtered, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFilterSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k_sample_filtered<<<rows, kFThreads, kFilterSmem, s>>>(p);
  return cudaGetLastError();
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
