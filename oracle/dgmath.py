"""fp32 exp and log used by the sampler, restated from textbook methods.

The sampler's decisions (argmax, the conf >= threshold test, the Gumbel-max
winner) are integers decided by floating point, so the oracle and the GPU
must take them with the same fp32 arithmetic.  Neither side may call its
platform's exp/log for that (they differ between libm and CUDA), so both
restate the same two functions from published methods, using only IEEE-754
single-precision +, -, *, / (each correctly rounded, no fused multiply-add)
and integer bit manipulation.

dg_exp(x)  -- Cody & Waite (1980) additive range reduction:
    k = floor(x * log2(e) + 1/2),  r = (x - k*C1) - k*C2
    with ln 2 split as C1 = 355/512 (exact in 9 bits, so k*C1 is exact) and
    C2 = fp32(ln 2 - C1); then the degree-7 Taylor polynomial of e^r
    (coefficients fp32(1/j!)) in Horner form, scaled by 2^k built from bits.
    Domain handling: NaN -> NaN, x < -87 -> 0, x > 88 -> +inf (so k stays in
    [-125, 127] and 2^k is a normal number).

dg_log(x)  -- exponent/mantissa split x = 2^e * m with m in [sqrt(1/2), sqrt(2)],
    then log m = 2 atanh(s), s = (m-1)/(m+1), by its odd series
    2(s + s^3/3 + ... + s^11/11) in Horner form over z = s^2, and
    log x = (e*C2 + log m) + e*C1 with the same ln 2 split.
    Domain: x <= 0 -> NaN (x == 0 -> -inf), +inf -> +inf, subnormals are
    pre-scaled by 2^23.

parity pinned by: tests/test_oracle_dgmath.py (libm in double as the exact
value: <= 2 ulp over the used ranges; exp(0) = 1, exp(-inf) = 0, log(1) = 0).
"""
import math

import numpy as np

f32 = np.float32

LOG2E = f32(1.0 / math.log(2.0))
LN2_HI = f32(355.0 / 512.0)                       # 0.693359375, 9 significant bits
LN2_LO = f32(math.log(2.0) - 355.0 / 512.0)
EXP_C = [f32(1.0 / math.factorial(j)) for j in range(8)]   # 1, 1, 1/2, ..., 1/5040
LOG_C = [f32(1.0 / j) for j in (3, 5, 7, 9, 11)]
SQRT2 = f32(math.sqrt(2.0))
EXP_LO = f32(-87.0)
EXP_HI = f32(88.0)


def dg_exp(x):
    x = np.asarray(x, dtype=f32)
    with np.errstate(invalid="ignore", over="ignore"):
        xc = np.clip(np.where(np.isnan(x), f32(0), x), EXP_LO, EXP_HI)
        t = xc * LOG2E
        kf = np.floor(t + f32(0.5))
        r = xc - kf * LN2_HI
        r = r - kf * LN2_LO
        p = EXP_C[7]
        for j in range(6, -1, -1):
            p = p * r + EXP_C[j]
        k = kf.astype(np.int32)
        scale = ((k + 127).astype(np.int32) << 23).view(f32)
        y = (p * scale).astype(f32)
    y = np.where(x < EXP_LO, f32(0), y)
    y = np.where(x > EXP_HI, f32(np.inf), y)
    y = np.where(np.isnan(x), x, y)
    return y.astype(f32)


def dg_log(x):
    x = np.asarray(x, dtype=f32)
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        sub = (x > 0) & (x < f32(2.0 ** -126))
        xs = np.where(sub, x * f32(2.0 ** 23), x).astype(f32)
        bits = xs.view(np.int32)
        e = ((bits >> 23) & 0xFF) - 127 - np.where(sub, 23, 0)
        m = ((bits & 0x7FFFFF) | 0x3F800000).view(f32)
        big = m > SQRT2
        m = np.where(big, m * f32(0.5), m).astype(f32)
        e = e + big.astype(np.int32)
        s = (m - f32(1.0)) / (m + f32(1.0))
        z = s * s
        q = LOG_C[4]
        for c in (LOG_C[3], LOG_C[2], LOG_C[1], LOG_C[0]):
            q = q * z + c
        q = q * z
        lm = s + s * q
        lm = lm + lm
        ef = e.astype(f32)
        r = ef * LN2_LO + lm
        r = r + ef * LN2_HI
    r = np.where(x == 0, f32(-np.inf), r)
    r = np.where(x < 0, f32(np.nan), r)
    r = np.where(np.isinf(x) & (x > 0), f32(np.inf), r)
    r = np.where(np.isnan(x), x, r)
    return r.astype(f32)


def gumbel_from_uniform(u):
    """Standard Gumbel noise g = -log(-log(u)) for u in (0, 1), in dg_log."""
    return -dg_log(-dg_log(u))
