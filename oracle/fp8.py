"""FP8 (e4m3) quantization of expert weights and expert inputs (oracle).

Test infrastructure only: imported by tests/, the package's smoke() and
bench.py's CPU legs; it shares nothing with the CUDA path.

The pages say only that serving ran with FP8 weights (blog "Test Conditions
Behind 1,456 Tokens per Second"); the format, the scaling and which operands
are quantized are not given.  Reading taken (stated in the design notes):

  * format: e4m3 without infinities ("fn"): 1 sign, 4 exponent bits (bias 7),
    3 mantissa bits, largest finite 448, subnormal step 2^-9; conversion
    rounds to nearest, ties to even, and saturates at +-448;
  * scaling: one power of two per row (an output feature of W_gate / W_up, or
    a token row of the expert input): the smallest k with
    max|row| <= 448 * 2^k, the row stored as e4m3(row * 2^-k);
  * what is quantized: the gate/up weights and their input rows; W_down and
    the SwiGLU output stay bf16.

parity pinned by: tests/test_oracle_fp8.py (e4m3 rounding equal to torch's
float8_e4m3fn conversion on every bf16 value within range; the scale rule's
bracketing property; the relative error bound of a quantized row).
"""
import numpy as np

E4M3_MAX = 448.0


def e4m3_round(v):
    """Values of e4m3(v): round to nearest even on the e4m3 grid, saturating
    at +-448 (float64 array in, float64 array out)."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    m, e = np.frexp(a)                       # a = m 2^e, m in [0.5, 1); floor(log2 a) = e - 1
    ex = np.maximum(e - 1, -6)               # normal exponent, or the subnormal range's
    quantum = np.ldexp(1.0, ex - 3)          # 3 mantissa bits
    q = np.rint(a / quantum) * quantum       # exact division by a power of two; rint: ties to even
    q = np.minimum(q, E4M3_MAX)
    q = np.where(a == 0, 0.0, q)
    return np.copysign(q, v)


def scale_exponent(absmax):
    """Smallest k with absmax <= 448 * 2^k (0 for absmax == 0), per element."""
    a = np.asarray(absmax, np.float64)
    m, e = np.frexp(a)                       # a = m 2^e; 448 * 2^(e-9) = 0.875 * 2^e
    k = np.where(m <= 0.875, e - 9, e - 8)
    return np.where(a == 0, 0, k).astype(np.int64)


def quantize_rows(w):
    """w [R, C] (values exact in float32) -> (q [R, C] e4m3 values, k [R]):
    row r is represented as q[r] * 2^k[r]."""
    w = np.asarray(w, np.float64)
    k = scale_exponent(np.max(np.abs(w), axis=1))
    q = e4m3_round(np.ldexp(w, -k[:, None]))
    return q, k


def dequantize_rows(q, k):
    return np.ldexp(np.asarray(q, np.float64), np.asarray(k)[:, None])


def e4m3_bits(q):
    """Bit patterns (uint8) of e4m3 values q (exactly representable)."""
    q = np.asarray(q, np.float64)
    sign = (np.signbit(q)).astype(np.uint8) << 7
    a = np.abs(q)
    m, e = np.frexp(a)                       # a = m 2^e
    ex = e - 1                               # floor(log2 a)
    normal = ex >= -6
    # normal: a = (1 + f/8) 2^ex, biased exponent ex + 7; subnormal: a = f 2^-9
    f_norm = np.rint((np.ldexp(a, -ex) - 1.0) * 8.0)
    f_sub = np.rint(np.ldexp(a, 9))
    bits = np.where(normal, ((ex + 7).astype(np.int64) << 3) | f_norm.astype(np.int64), f_sub.astype(np.int64))
    bits = np.where(a == 0, 0, bits)
    return (bits.astype(np.uint8) | sign)
