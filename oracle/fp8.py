"""8-bit floating-point KV storage (e4m3) — TEST INFRASTRUCTURE.

kgptalkie "Day 28: PagedAttention / vLLM", "Split the Cache Into Fixed Blocks":
the bytes of a block depend on the number of heads, the head width and the
dtype.  The fp8 pool variant keeps each key and value element as one byte:

* format e4m3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent
  field 0 is subnormal (value m * 2^-9), the all-ones exponent with mantissa
  7 is NaN, and there is no infinity: the largest finite magnitude is 448;
* quantizing (this build's reading; the pages name the dtype only): a value
  x of the appended token (bf16) is divided by the pool's fp32 scale in IEEE
  float32, y = fl32(x / scale), and y is rounded to the nearest e4m3 value,
  ties to the even code, magnitudes beyond 448 saturating to 448;
* a stored code c means decode(c) * scale.

Written from the format's definition, in float64 (every e4m3 value and every
float32 is exact there).
"""
import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 code (uint8 array) as float64; NaN codes give NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def e4m3_encode(y) -> np.ndarray:
    """Nearest e4m3 code to each float32 value y (ties to the even code),
    magnitudes beyond 448 saturating to 448; NaN gives the NaN code 0x7F."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    nan = np.isnan(y)
    neg = np.signbit(y)
    a = np.abs(np.where(nan, 0.0, y))
    a = np.minimum(a, E4M3_MAX)
    # exponent of the binade: normal e4m3 binades are 2^-6 .. 2^8, each with
    # 8 steps of 2^(e-3); below 2^-6 the step is 2^-9 (subnormal)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    # frexp-exact binade: correct floor(log2) if it is off by one at a power of two
    e = np.where(a >= np.exp2(e + 1), e + 1, e)
    e = np.where((a < np.exp2(e)) & (e > -6), e - 1, e)
    step = np.exp2(e - 3)
    q = np.rint(a / step) * step                  # a / step is exact; rint ties to even
    q = np.minimum(q, E4M3_MAX)
    # encode q
    sub = q < 2.0 ** -6
    m_sub = np.rint(q / 2.0 ** -9).astype(np.int64)                # 0..7 (8 would be normal)
    eq = np.floor(np.log2(np.where(q > 0, q, 1.0))).astype(np.int64)
    m_nrm = np.rint(q / np.exp2(eq - 3.0)).astype(np.int64) - 8    # 0..7
    code = np.where(sub, m_sub, ((eq + 7) << 3) | m_nrm)
    code = np.where(neg, code | 0x80, code)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def quantize(x, scale) -> np.ndarray:
    """Codes of the values x (any float array; bf16/fp32 values widen exactly)
    for a pool scale: e4m3_encode(fl32(x / scale))."""
    y = np.asarray(x, dtype=np.float32) / np.float32(scale)      # IEEE float32 division
    return e4m3_encode(y)


def dequantize(codes, scale) -> np.ndarray:
    """float64 values decode(c) * scale (exact: 4-bit times 24-bit significands)."""
    return e4m3_decode(codes) * float(np.float32(scale))
