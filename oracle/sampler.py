"""On-device sampling restated on the CPU -- TEST INFRASTRUCTURE.

"19. Fast decode", §Sampling without the CPU: with temperature 0 the step takes
the argmax of the logits; otherwise it adds Gumbel noise g = -log(-log u),
u ~ Uniform(0, 1), to logits / temperature and takes the argmax, which draws
exactly from softmax(logits / temperature) with elementwise work only.

The pages draw u with an unseeded generator and clamp it to [1e-10, 1].  The
build needs the same u on the CPU and the GPU, so the readings are:
  * u comes from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
    numbers: as easy as 1, 2, 3", SC 2011), key = (seed_lo, seed_hi), counter =
    (v >> 2, r, offset_lo, offset_hi) for request row r and vocabulary entry v,
    output word v & 3;
  * u = (2 * (x >> 9) + 1) * 2^-24 for the 32-bit word x: 2^23 evenly spaced
    values strictly inside (0, 1), each exact in float32, so no clamp is needed;
  * log is this module's own float32 routine (``ln_f32``) built from correctly
    rounded +, -, *, / only, so that both sides round identically;
  * z * (1 / T) + g is formed with two separately rounded float32 operations,
    1 / T in float32; ties of the maximum go to the lowest index.

Parity: Philox is pinned against Triton's Philox run on the CPU interpreter and
by uniformity checks; ln_f32 against libm within 2 ulp; the sampler against an
independent float64 argmax of z + g and by a chi-squared test of 20,000 draws
("19. Fast decode", §Sampling without the CPU: the milestone test).
"""
from __future__ import annotations

import math

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten rounds of Philox4x32 on counter (c0..c3) under key (k0, k1); arrays broadcast.

    Each round multiplies c0 and c2 by the two round multipliers, keeps the high
    and low 32-bit halves, mixes the high halves with the odd words and the key,
    and then bumps the key by the two Weyl constants (SC 2011, §Philox).
    """
    c0 = np.asarray(c0, dtype=np.uint64) & _MASK32
    c1 = np.asarray(c1, dtype=np.uint64) & _MASK32
    c2 = np.asarray(c2, dtype=np.uint64) & _MASK32
    c3 = np.asarray(c3, dtype=np.uint64) & _MASK32
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK32
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK32
    for _ in range(10):
        p0 = _M0 * c0
        p1 = _M1 * c2
        n0 = ((p1 >> np.uint64(32)) ^ c1 ^ k0) & _MASK32
        n1 = p1 & _MASK32
        n2 = ((p0 >> np.uint64(32)) ^ c3 ^ k1) & _MASK32
        n3 = p0 & _MASK32
        c0, c1, c2, c3 = n0, n1, n2, n3
        k0 = (k0 + _W0) & _MASK32
        k1 = (k1 + _W1) & _MASK32
    return (c0.astype(np.uint32), c1.astype(np.uint32), c2.astype(np.uint32), c3.astype(np.uint32))


def random_words(seed: int, offset: int, row: int, vocab: int) -> np.ndarray:
    """The 32-bit Philox word for every vocabulary entry of one request row."""
    v = np.arange(vocab, dtype=np.uint64)
    blocks = np.arange((vocab + 3) // 4, dtype=np.uint64)
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    offset = int(offset) & 0xFFFFFFFFFFFFFFFF
    out = philox4x32_10(blocks, row, offset & 0xFFFFFFFF, offset >> 32, seed & 0xFFFFFFFF, seed >> 32)
    words = np.stack(out, axis=1).reshape(-1)        # word 4*b + lane
    return words[v.astype(np.int64)]


def uniforms(seed: int, offset: int, row: int, vocab: int) -> np.ndarray:
    """u in (0, 1) as float32: (2 * (x >> 9) + 1) * 2^-24."""
    x = random_words(seed, offset, row, vocab)
    k = ((x >> np.uint32(9)).astype(np.int64) * 2 + 1).astype(np.float32)
    return k * np.float32(2.0 ** -24)


# --- float32 natural logarithm from correctly rounded operations only ----------------------------
#
# x = m * 2^e with m in [sqrt(1/2), sqrt(2)); ln x = e ln2 + ln m, and
# ln m = 2 atanh(s) = 2 (s + s^3/3 + s^5/5 + s^7/7 + s^9/9 + ...), s = (m-1)/(m+1),
# |s| <= 0.1716, so the truncated series is accurate far below float32 precision.
# ln2 is split into a short high part (exact when multiplied by |e| < 256) and a
# low part (Cody and Waite's argument-reduction technique).

_F = np.float32
_LN2 = math.log(2.0)
_LN2_HI = np.array([_LN2], dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFF000)
_LN2_HI = _LN2_HI.view(np.float32)[0]
_LN2_LO = _F(_LN2 - float(_LN2_HI))
_C3, _C5, _C7, _C9 = _F(1.0 / 3.0), _F(1.0 / 5.0), _F(1.0 / 7.0), _F(1.0 / 9.0)
_SQRT2_BITS = np.array([math.sqrt(2.0)], dtype=np.float32).view(np.uint32)[0]


def ln_constants() -> dict:
    """The float32 constants of ln_f32 as bit patterns (documented for cross-checks)."""
    as_bits = lambda f: int(np.array([f], dtype=np.float32).view(np.uint32)[0])
    return {"ln2_hi": as_bits(_LN2_HI), "ln2_lo": as_bits(_LN2_LO), "c3": as_bits(_C3), "c5": as_bits(_C5),
            "c7": as_bits(_C7), "c9": as_bits(_C9), "sqrt2": int(_SQRT2_BITS)}


def ln_f32(x) -> np.ndarray:
    """Natural log of positive normal float32 values, every step one rounded float32 operation."""
    x = np.asarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    e = (bits >> np.uint32(23)).astype(np.int32) - 127
    mbits = (bits & np.uint32(0x7FFFFF)) | np.uint32(0x3F800000)
    big = mbits > _SQRT2_BITS
    mbits = np.where(big, mbits - np.uint32(0x800000), mbits)   # m / 2, exact
    e = np.where(big, e + 1, e)
    m = mbits.view(np.float32)
    num = m - _F(1.0)
    den = m + _F(1.0)
    s = num / den
    z = s * s
    t = z * _C9
    t = t + _C7
    t = t * z
    t = t + _C5
    t = t * z
    t = t + _C3
    t = t * z
    r = s * t
    r = s + r
    r = r + r
    ef = e.astype(np.float32)
    a = ef * _LN2_LO
    a = a + r
    b = ef * _LN2_HI
    return b + a


def gumbel_f32(u) -> np.ndarray:
    """g = -ln(-ln u) in float32 with ``ln_f32``."""
    a = ln_f32(u)
    return -ln_f32(-a)


def sample_row(z: np.ndarray, temperature: float, seed: int, offset: int, row: int) -> int:
    """Sampled id for one row of float32 logits: greedy at temperature 0, Gumbel-max otherwise."""
    z = np.asarray(z, dtype=np.float32)
    if temperature == 0.0:
        return int(np.argmax(z))
    inv_t = _F(1.0) / _F(temperature)
    g = gumbel_f32(uniforms(seed, offset, row, z.shape[0]))
    key = (z * inv_t) + g
    return int(np.argmax(key))


def sample(logits: np.ndarray, temperatures, seed: int, offset: int) -> np.ndarray:
    """Sampled ids [R] for float32 logits [R, V]; row r uses Philox row r."""
    logits = np.asarray(logits, dtype=np.float32)
    temps = np.broadcast_to(np.asarray(temperatures, dtype=np.float64), (logits.shape[0],))
    return np.array([sample_row(logits[r], float(temps[r]), seed, offset, r) for r in range(logits.shape[0])],
                    dtype=np.int32)
