// sampling.cuh -- on-device Gumbel-max / greedy sampling arithmetic.
//
// "19. Fast decode", section "Sampling without the CPU": greedy argmax at temperature 0, otherwise the
// argmax of logits / T + g with g = -log(-log u), u ~ Uniform(0, 1), which draws from softmax(logits / T)
// with elementwise work only.  u comes from Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC 2011) so that any row / vocabulary entry can be regenerated:
// key = (seed_lo, seed_hi), counter = (v >> 2, r, offset_lo, offset_hi), word v & 3, and
// u = (2 * (x >> 9) + 1) * 2^-24, strictly inside (0, 1).
//
// The logarithm is computed here from correctly rounded float32 +, -, *, / only (explicit _rn
// intrinsics, which the compiler never fuses), so a CPU restatement with the same operation order
// reproduces every bit: x = m 2^e with m in [sqrt(1/2), sqrt(2)), ln m = 2 atanh(s) with
// s = (m - 1) / (m + 1) summed to s^9 / 9, ln 2 split into a short high part and a low part.
#pragma once

#include "common.cuh"

namespace grd {

struct Philox4 {
  uint32_t x[4];
};

ENG_DEVICE Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
    const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += W0;
    k1 += W1;
  }
  Philox4 r;
  r.x[0] = c0;
  r.x[1] = c1;
  r.x[2] = c2;
  r.x[3] = c3;
  return r;
}

ENG_DEVICE float uniform_from_word(uint32_t x) {
  const int k = (int)(x >> 9) * 2 + 1;  // < 2^24: exact in float32
  return __fmul_rn(__int2float_rn(k), 5.9604644775390625e-08f /* 2^-24 */);
}

ENG_DEVICE float philox_uniform(uint32_t seed_lo, uint32_t seed_hi, uint32_t off_lo, uint32_t off_hi, uint32_t row,
                                uint32_t v) {
  const Philox4 p = philox4x32_10(v >> 2, row, off_lo, off_hi, seed_lo, seed_hi);
  const uint32_t w = p.x[v & 3];
  return uniform_from_word(w);
}

// Float32 constants of the logarithm: ln 2 with its low 12 mantissa bits cleared, the remainder, the
// series coefficients 1/3, 1/5, 1/7, 1/9 rounded to float32, and sqrt(2) rounded to float32.
#define ENG_LN2_HI_BITS 0x3F317000u
#define ENG_SQRT2_BITS 0x3FB504F3u

ENG_DEVICE float ln_f32(float x) {
  const float ln2_hi = __uint_as_float(ENG_LN2_HI_BITS);
  const float ln2_lo = __uint_as_float(0x3805FDF4u);  // float32(ln 2 - ln2_hi)
  const float c3 = __uint_as_float(0x3EAAAAABu);      // float32(1/3)
  const float c5 = __uint_as_float(0x3E4CCCCDu);      // float32(1/5)
  const float c7 = __uint_as_float(0x3E124925u);      // float32(1/7)
  const float c9 = __uint_as_float(0x3DE38E39u);      // float32(1/9)
  const uint32_t bits = __float_as_uint(x);
  int e = (int)(bits >> 23) - 127;
  uint32_t mb = (bits & 0x7FFFFFu) | 0x3F800000u;
  if (mb > ENG_SQRT2_BITS) {
    mb -= 0x800000u;  // m / 2, exact
    e += 1;
  }
  const float m = __uint_as_float(mb);
  const float num = __fsub_rn(m, 1.0f);
  const float den = __fadd_rn(m, 1.0f);
  const float s = __fdiv_rn(num, den);
  const float z = __fmul_rn(s, s);
  float t = __fmul_rn(z, c9);
  t = __fadd_rn(t, c7);
  t = __fmul_rn(t, z);
  t = __fadd_rn(t, c5);
  t = __fmul_rn(t, z);
  t = __fadd_rn(t, c3);
  t = __fmul_rn(t, z);
  float r = __fmul_rn(s, t);
  r = __fadd_rn(s, r);
  r = __fadd_rn(r, r);
  const float ef = __int2float_rn(e);
  float a = __fmul_rn(ef, ln2_lo);
  a = __fadd_rn(a, r);
  const float b = __fmul_rn(ef, ln2_hi);
  return __fadd_rn(b, a);
}

ENG_DEVICE float gumbel_from_uniform(float u) {
  const float a = ln_f32(u);
  return -ln_f32(-a);
}

// Sampling key of one logit: z (greedy) or z * inv_t + g, each a separately rounded float32 operation.
ENG_DEVICE float sample_key(float z, float inv_t, const uint32_t rng[4], uint32_t row, uint32_t v) {
  if (inv_t == 0.0f) return z;
  const float u = philox_uniform(rng[0], rng[1], rng[2], rng[3], row, v);
  const float g = gumbel_from_uniform(u);
  return __fadd_rn(__fmul_rn(z, inv_t), g);
}

// Orders (key, index) pairs as one unsigned 64-bit integer: larger key first, then lower index.
ENG_DEVICE unsigned long long pack_key_index(float key, uint32_t index) {
  const uint32_t f = __float_as_uint(key);
  const uint32_t ord = (f & 0x80000000u) ? ~f : (f | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(~index);
}

ENG_DEVICE uint32_t unpack_index(unsigned long long packed) { return ~(uint32_t)(packed & 0xFFFFFFFFull); }

}  // namespace grd
