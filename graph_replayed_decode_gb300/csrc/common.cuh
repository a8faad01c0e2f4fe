// common.cuh -- shared device helpers of libeng: 16-bit element packing, warp reductions and thin
// inline-PTX wrappers (warp-level MMA, ldmatrix, cp.async, programmatic dependent launch).
//
// Element type.  Weights, the K/V cache and the operand planes are 16-bit values held in the storage
// type bf16.  The kernel files whose arithmetic depends on the format (gemm.cu, attn_decode.cu,
// attn_prefill.cu, norm.cu, pack.cu) are compiled twice: as they stand for bfloat16, and with ENG_F16
// defined for IEEE binary16 (the fp16 variant of a model), into the nested namespace grd::f16.  In an
// ENG_F16 translation unit the bits in bf16 storage are binary16 values, and every conversion and MMA
// below reads and writes them as such; no kernel converts between the formats.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;

#ifdef ENG_F16
#define ENG_ELEM_NS_BEGIN namespace f16 {
#define ENG_ELEM_NS_END }
#else
#define ENG_ELEM_NS_BEGIN
#define ENG_ELEM_NS_END
#endif

#define ENG_DEVICE __device__ __forceinline__

// ------------------------------------------------------------------ status word bits (mirror eng.h)
#define ST_BAD_BLOCK 1
#define ST_BAD_POSITION 2
#define ST_NAN 4
#define ST_TIMEOUT 8

ENG_DEVICE void set_status(int* status, int bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------------------------ 16-bit element helpers
// (static: an ENG_F16 translation unit defines them for binary16; each unit keeps its own)
#ifdef ENG_F16
static ENG_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

static ENG_DEVICE float2 unpack_bf16x2(uint32_t u) {
  __half2 v = *reinterpret_cast<__half2*>(&u);
  return __half22float2(v);
}

static ENG_DEVICE float elem_to_float(bf16 x) { return __half2float(*reinterpret_cast<const __half*>(&x)); }

static ENG_DEVICE bf16 float_to_elem(float v) {
  const __half h = __float2half_rn(v);
  return *reinterpret_cast<const bf16*>(&h);
}
#else
static ENG_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

static ENG_DEVICE float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

static ENG_DEVICE float elem_to_float(bf16 x) { return __bfloat162float(x); }

static ENG_DEVICE bf16 float_to_elem(float v) { return __float2bfloat16_rn(v); }
#endif

ENG_DEVICE float bf16_bits_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Activation operands of the tensor-core products are carried as bf16 pairs: hi = bf16(v) and
// lo = bf16(v - hi) (the difference is exact in fp32), so hi + lo keeps about 16 significant bits and a
// product over the pair (W.hi + W.lo, accumulated in fp32) loses almost nothing to operand rounding.
// Single-bf16 activations would put every projection's input through a 2^-9 rounding, and over a few
// dozen layers that alone moves the logits by several hundredths.  (Binary16 pairs keep about 22 bits
// where the low half stays a normal number; below 2^-14 it loses bits to the format's narrow range.)
static ENG_DEVICE void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  const float2 hf = unpack_bf16x2(hi);
  lo = pack_bf16x2(a - hf.x, b - hf.y);
}

// One value into the operand planes at element index i.
static ENG_DEVICE void put_split(bf16* xh, bf16* xl, size_t i, float v) {
  const bf16 h = float_to_elem(v);
  xh[i] = h;
  xl[i] = float_to_elem(v - elem_to_float(h));
}

// Two adjacent values (i even) into the operand planes.
static ENG_DEVICE void put_split2(bf16* xh, bf16* xl, size_t i, float a, float b) {
  uint32_t h, l;
  split_bf16x2(a, b, h, l);
  *reinterpret_cast<uint32_t*>(xh + i) = h;
  *reinterpret_cast<uint32_t*>(xl + i) = l;
}

// ------------------------------------------------------------------ reductions (fixed xor trees)
ENG_DEVICE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

ENG_DEVICE float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------------ loads
// Streaming 16-byte load that bypasses L1 allocation (weights are read once per step).
ENG_DEVICE uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

ENG_DEVICE uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

ENG_DEVICE void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src));
}
// The same with an L2 cache policy for the source line.
ENG_DEVICE void cp_async16_hint(void* smem_dst, const void* gmem_src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src),
               "l"(pol));
}
ENG_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
ENG_DEVICE void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

// ------------------------------------------------------------------ L2 cache policies
// Data read once per step and never again in it (the K/V stream) is marked evict-first; weights
// prefetched into L2 for a later kernel are marked evict-last, so that a large K/V stream in between
// does not push them out.
ENG_DEVICE uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
ENG_DEVICE uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ------------------------------------------------------------------ L2 prefetch
ENG_DEVICE void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
ENG_DEVICE void prefetch_l2_keep(const void* p, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(pol)
               : "memory");
}

// This CTA's share of an L2 prefetch of `bytes` (a multiple of 16) at p, split evenly over the grid.
ENG_DEVICE void prefetch_share(const void* p, unsigned long long bytes) {
  const unsigned long long ctas = (unsigned long long)gridDim.x * gridDim.y * gridDim.z;
  const unsigned long long id = blockIdx.x + (unsigned long long)gridDim.x * (blockIdx.y + (unsigned long long)gridDim.y * blockIdx.z);
  const unsigned long long share = ((bytes + ctas - 1) / ctas + 15) & ~15ull;
  unsigned long long lo = id * share, hi = lo + share;
  if (hi > bytes) hi = bytes;
  const uint64_t pol = l2_evict_last();
  for (unsigned long long o = lo; o < hi; o += 65536) {
    const unsigned long long n = hi - o < 65536 ? hi - o : 65536;
    prefetch_l2_keep(static_cast<const char*>(p) + o, (uint32_t)n, pol);
  }
}

// ------------------------------------------------------------------ TMA bulk copies and mbarriers
// One mbarrier tracks the bytes of the bulk copies issued against it; waits are bounded.
ENG_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

ENG_DEVICE void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from global to this CTA's shared
// memory, completing on `bar`.
ENG_DEVICE void tma_load_1d(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Waits for phase `parity` of the barrier to complete; gives up after `limit` polls and returns false.
ENG_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// ------------------------------------------------------------------ TMA tensor copies and 5th-gen tensor cores
// A 2D tiled bulk copy of box (x, y) of `map` (128-byte swizzled rows) into shared memory (1024-byte aligned),
// completing on `bar`.  x is the innermost coordinate in elements (a multiple of 64 here).
ENG_DEVICE void tma_tile_2d(void* smem_dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile whose rows are 128 bytes (64 bf16) with the 128-byte
// swizzle a TMA tensor copy applies: 8-row groups 1024 bytes apart (stride byte offset), swizzle mode 2,
// descriptor version 1.  Adding 2 advances the start by 32 bytes, i.e. 16 elements along K.
ENG_DEVICE uint64_t umma_desc_sw128(const void* tile) {
  const uint64_t a = smem_u32(tile);
  return ((a & 0x3FFFF) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the element type (format code 1 for
// bf16, 0 for binary16 -- both operands alike), both K-major, M x N.
#ifdef ENG_F16
static constexpr uint32_t kUmmaAbFormat = 0u;
#else
static constexpr uint32_t kUmmaAbFormat = 1u;
#endif
static __host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (kUmmaAbFormat << 7) | (kUmmaAbFormat << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A . B^T, issued by one thread.
ENG_DEVICE void umma_bf16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tensor-core operation issued so far by this thread has completed.
ENG_DEVICE void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Tensor-memory columns for this CTA (a power of two >= 32), address written to *dst by the warp.
template <int NCOLS>
ENG_DEVICE void tmem_alloc(uint32_t* dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "n"(NCOLS)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <int NCOLS>
ENG_DEVICE void tmem_free(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(NCOLS) : "memory");
}

ENG_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
ENG_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread) from address taddr.
ENG_DEVICE void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// ------------------------------------------------------------------ warp MMA (m16n8k16, 16-bit in, f32 accumulate)
// A: 16x16 row-major fragment (4 regs), B: 16x8 column fragment (2 regs), C/D: 16x8 f32 (4 regs); A and B
// of the element type (bf16, or binary16 in an ENG_F16 unit).
#ifdef ENG_F16
#define ENG_MMA_TYPES "f16.f16"
#else
#define ENG_MMA_TYPES "bf16.bf16"
#endif
static ENG_DEVICE void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32." ENG_MMA_TYPES ".f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

ENG_DEVICE void ldmatrix_x4(uint32_t r[4], const void* smem_row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(smem_row_addr)));
}

ENG_DEVICE void ldmatrix_x4_trans(uint32_t r[4], const void* smem_row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(smem_row_addr)));
}

// ------------------------------------------------------------------ programmatic dependent launch
// Wait until the preceding kernel in the stream has completed and its writes are visible.  A no-op
// when the kernel was launched without the programmatic-serialisation attribute.
ENG_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to begin launching (its own pdl_wait still orders its reads).
ENG_DEVICE void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// ------------------------------------------------------------------ packed weight layout
// A weight matrix W[N][K] (row-major, N % 16 == 0, K % 32 == 0) is stored as tiles of 16 rows x 32
// columns, tile (i, j) at ((i * K/32) + j) * 512 elements.  Inside a tile the 512 values are ordered
// [k-step s (2)][lane (32)][8] so that one 16-byte load per lane yields that lane's m16n8k16 A
// fragment for k-step s: with g = lane / 4, t = lane % 4, the 8 values are
//   W[16i+g][32j+16s+2t+{0,1}], W[16i+g+8][..same..], W[16i+g][32j+16s+2t+8+{0,1}], W[16i+g+8][..same..].
ENG_DEVICE size_t packed_offset(int row, int col, int K) {
  const int i = row >> 4, r = row & 15;
  const int j = col >> 5, kk = col & 31;
  const int s = kk >> 4, kr = kk & 15;
  const int g = r & 7, half = r >> 3;
  const int hi8 = kr >> 3, t = (kr & 7) >> 1, lo = kr & 1;
  const int lane = g * 4 + t;
  const int e = hi8 * 4 + half * 2 + lo;
  return ((size_t)i * (K >> 5) + j) * 512 + (size_t)s * 256 + lane * 8 + e;
}
