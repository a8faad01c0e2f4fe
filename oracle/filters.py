"""Top-k and top-p filtering ahead of the Gumbel-max draw -- TEST INFRASTRUCTURE.

"19. Fast decode", §Sampling without the CPU: both filters run before the
argmax by setting the filtered logits to -inf; a fixed k keeps the shapes
static, and top-p does too when it is a sort and a mask instead of a slice.
The pages name the filters but do not define them, so this module takes the
usual definitions and fixes every step that decides an integer:

  * rank order: logits by value, larger first; equal values (+0 and -0 are
    equal) in increasing index order;
  * top-k keeps the first k entries of the rank order (k <= 0 or k >= V: off);
  * temperature first: s = z * (1/T) in float32, as the unfiltered sampler
    forms it; top-p then works on softmax(s) over the top-k survivors
    (renormalised among them);
  * top-p keeps the shortest prefix of the rank order whose probability mass
    reaches p (0 < p < 1; otherwise off), so the top entry always survives;
  * the probabilities are taken in exact integer arithmetic so that the cut
    does not depend on a summation order: e_v = exp_f32(s_v - s_max) (this
    module's own float32 exp, below), weight w_v = floor(e_v * 2^32), p as
    P = max(1, rint(p * 2^24)) in units of 2^-24, and entry v survives iff
    C_v * 2^24 < P * W, where C_v is the weight of the survivors ahead of v and
    W the total; equivalently C_v <= (P * W - 1) >> 24;
  * the draw is the unfiltered sampler's key s + g (Philox noise, float32),
    argmax over the survivors, ties to the lowest index; temperature 0 stays
    the plain argmax (neither filter can drop the top entry).

Parity: exp_f32 is pinned against libm within 2 ulp over its whole range; the
integer cut against brute force and against dyadic distributions whose
nucleus is known in closed form; the filters' special cases against the
pinned unfiltered sampler and torch.topk; the draws by chi-squared tests
against the filtered softmax.
"""
from __future__ import annotations

import math

import numpy as np

from .sampler import gumbel_f32, uniforms

_F = np.float32

# --- float32 exp from correctly rounded operations only -------------------------------------------
#
# exp(d) = 2^n * exp(r) with n = rint(d / ln 2) and r = d - n ln 2, |r| <= ln2 / 2 (Cody and Waite's
# reduction, ln 2 split into a 12-bit high part -- exact when multiplied by |n| < 2^12 -- and a low part);
# exp(r) by its Taylor series to r^7 / 7! (truncation below 6e-9 relative) in Horner form; 2^n exactly
# from the exponent bits.  Only d in [-23, 0] is needed: exp(-23) < 2^-32, whose weight is 0 anyway.

_INV_LN2 = _F(1.0 / math.log(2.0))
_LN2_HI = (np.array([math.log(2.0)], dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFF000)).view(np.float32)[0]
_LN2_LO = _F(math.log(2.0) - float(_LN2_HI))
_EXP_C = [_F(1.0 / math.factorial(k)) for k in range(8)]      # 1, 1, 1/2, ..., 1/7!
EXP_MIN = _F(-23.0)


def exp_constants() -> dict:
    """The float32 constants of exp_f32 as bit patterns (documented for cross-checks)."""
    as_bits = lambda f: int(np.array([f], dtype=np.float32).view(np.uint32)[0])
    out = {"inv_ln2": as_bits(_INV_LN2), "ln2_hi": as_bits(_LN2_HI), "ln2_lo": as_bits(_LN2_LO)}
    out.update({f"c{k}": as_bits(c) for k, c in enumerate(_EXP_C)})
    return out


def exp_f32(d) -> np.ndarray:
    """e^d for float32 d <= 0, every step one rounded float32 operation; 0 below -23."""
    d = np.asarray(d, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore"):       # far below -23 the result is replaced by 0
        n = np.rint(d * _INV_LN2)                                # rint: ties to even, exact
        r = d - n * _LN2_HI
        r = r - n * _LN2_LO
        p = _EXP_C[7]
        for k in range(6, -1, -1):
            p = p * r
            p = p + _EXP_C[k]
        ni = np.clip(np.nan_to_num(n), -126, 127).astype(np.int32)
        scale = ((ni + 127).astype(np.uint32) << np.uint32(23)).view(np.float32)
        out = p * scale
    return np.where(d < EXP_MIN, _F(0.0), out).astype(np.float32)


# --- the filters ---------------------------------------------------------------------------------

def rank_order(z: np.ndarray) -> np.ndarray:
    """Indices of z by value, larger first, equal values in increasing index order."""
    z = np.asarray(z, dtype=np.float32)
    return np.lexsort((np.arange(z.shape[0]), -z.astype(np.float64)))


def p_units(top_p: float) -> int:
    """top_p in units of 2^-24: P = max(1, rint(p * 2^24)); 0 means no top-p filter (p <= 0 or p >= 1)."""
    p = _F(top_p)
    if not (p > 0.0 and p < 1.0):
        return 0
    P = int(np.rint(p * _F(2.0 ** 24)))
    return 0 if P >= 2 ** 24 else max(1, P)


def nucleus_weights(s_ranked: np.ndarray, s_max) -> np.ndarray:
    """w = floor(exp_f32(s - s_max) * 2^32) as int64, for float32 s in rank order."""
    e = exp_f32(np.asarray(s_ranked, dtype=np.float32) - _F(s_max))
    return np.floor(e.astype(np.float64) * 2.0 ** 32).astype(np.int64)


def nucleus_size(w_ranked: np.ndarray, P: int) -> int:
    """How many entries, in rank order, survive top-p: those with C_v * 2^24 < P * W (C_v = mass ahead)."""
    w = [int(x) for x in w_ranked]
    W = sum(w)
    ahead, n = 0, 0
    for x in w:
        if ahead * 2 ** 24 < P * W:
            n += 1
        else:
            break                                                # C_v only grows along the rank order
        ahead += x
    return n


def survivors(z: np.ndarray, temperature: float, top_k: int, top_p: float) -> np.ndarray:
    """Sorted indices of the entries that survive both filters (temperature > 0)."""
    z = np.asarray(z, dtype=np.float32)
    V = z.shape[0]
    inv_t = _F(1.0) / _F(temperature)
    s = z * inv_t
    order = rank_order(z)
    keep = order if (top_k <= 0 or top_k >= V) else order[:top_k]
    P = p_units(top_p)
    if P:
        w = nucleus_weights(s[keep], s[order[0]])
        keep = keep[:nucleus_size(w, P)]
    return np.sort(keep)


def sample_row_filtered(z: np.ndarray, temperature: float, top_k: int, top_p: float, seed: int, offset: int,
                        row: int) -> int:
    """One draw: argmax of s + g over the survivors (temperature > 0), or the plain argmax (temperature 0)."""
    z = np.asarray(z, dtype=np.float32)
    if temperature == 0.0:
        return int(np.argmax(z))
    inv_t = _F(1.0) / _F(temperature)
    keep = survivors(z, temperature, top_k, top_p)
    key = (z * inv_t) + gumbel_f32(uniforms(seed, offset, row, z.shape[0]))
    masked = np.full(z.shape[0], -np.inf, dtype=np.float32)
    masked[keep] = key[keep]
    return int(np.argmax(masked))


def sample_filtered(logits: np.ndarray, temperatures, top_k, top_p, seed: int, offset: int) -> np.ndarray:
    """Sampled ids [R] for float32 logits [R, V] with per-row temperature, top-k and top-p."""
    logits = np.asarray(logits, dtype=np.float32)
    R = logits.shape[0]
    t = np.broadcast_to(np.asarray(temperatures, dtype=np.float64), (R,))
    k = np.broadcast_to(np.asarray(top_k, dtype=np.int64), (R,))
    p = np.broadcast_to(np.asarray(top_p, dtype=np.float64), (R,))
    return np.array([sample_row_filtered(logits[r], float(t[r]), int(k[r]), float(p[r]), seed, offset, r)
                     for r in range(R)], dtype=np.int32)


def survivor_counts(logits: np.ndarray, temperatures, top_k, top_p) -> np.ndarray:
    """Number of survivors per row (1 at temperature 0: the argmax)."""
    logits = np.asarray(logits, dtype=np.float32)
    R = logits.shape[0]
    t = np.broadcast_to(np.asarray(temperatures, dtype=np.float64), (R,))
    k = np.broadcast_to(np.asarray(top_k, dtype=np.int64), (R,))
    p = np.broadcast_to(np.asarray(top_p, dtype=np.float64), (R,))
    return np.array([1 if t[r] == 0.0 else len(survivors(logits[r], float(t[r]), int(k[r]), float(p[r])))
                     for r in range(R)], dtype=np.int32)
