"""Bit-level codecs for the two storage formats the fused operators read and write.

Test infrastructure only: nothing in the product path imports this package.

Both codecs are written from the format definitions, with numpy doing plain
float64 arithmetic on the fields:

* bfloat16 -- 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits; the
  upper half of an IEEE binary32.  Encoding rounds to nearest, ties to an even
  fraction, overflows to +-inf, and keeps subnormals (step 2**-133).
* OCP FP8 E4M3 ("fn" variant) -- 1 sign bit, 4 exponent bits (bias 7),
  3 fraction bits, no infinities, S.1111.111 is NaN, largest finite value 448,
  subnormals m * 2**-9.  The fused RMSNorm kernel of the FlashRT page
  ("FlashRT 跨层融合深度解析", §2.1 and §3) writes its activations in this
  format; the clamp-before-encode rule follows the OpenPPL page
  ("OpenPPL算子融合深度解析", §6.4: a fused clamp must see the quantisation
  scale), read here as saturation to +-448 instead of overflow to NaN.
"""
import numpy as np

# ----------------------------------------------------------------- bfloat16

BF16_EXP_BIAS = 127
BF16_FRAC_BITS = 7
BF16_MIN_NORMAL_EXP = -126          # 2**-126 is the smallest normal
BF16_SUB_STEP_EXP = -133            # subnormal spacing 2**-126 / 2**7


def bf16_decode(bits):
    """uint16 bit patterns -> float64 values, from the sign/exponent/fraction fields."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    f = (b & 0x7F).astype(np.float64)
    normal = np.ldexp(1.0 + f / 128.0, (e - BF16_EXP_BIAS).astype(np.int32))
    sub = np.ldexp(f, BF16_SUB_STEP_EXP)
    val = np.where(e == 0, sub, normal)
    val = np.where(e == 0xFF, np.where(f == 0, np.inf, np.nan), val)
    return sign * val


def bf16_encode(x):
    """float64 values -> uint16 bfloat16 bits, round to nearest even, one rounding."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64)
    a = np.abs(x)
    with np.errstate(invalid="ignore", over="ignore"):
        # Normal range: a = (1 + q/128) * 2**e with e = floor(log2 a).
        mant, ex = np.frexp(a)                       # a = mant * 2**ex, mant in [0.5, 1)
        e = ex.astype(np.int64) - 1
        q = np.rint((2.0 * mant - 1.0) * 128.0)      # rint: ties to even
        carry = q >= 128.0
        e = np.where(carry, e + 1, e)
        q = np.where(carry, 0.0, q)
        normal_bits = ((e + BF16_EXP_BIAS) << 7) | q.astype(np.int64)
        overflow = e > 127
        normal_bits = np.where(overflow, 0xFF << 7, normal_bits)
        # Subnormal range: a = q * 2**-133 (q = 128 lands on the smallest normal).
        qs = np.rint(np.ldexp(a, -BF16_SUB_STEP_EXP)).astype(np.int64)
        is_sub = a < np.ldexp(1.0, BF16_MIN_NORMAL_EXP)
        bits = np.where(is_sub, qs, normal_bits)
        bits = np.where(np.isinf(a), 0xFF << 7, bits)
        bits = np.where(np.isnan(a), 0x7FC0, bits | (sign << 15))
    return bits.astype(np.uint16)


def bf16_round(x):
    """Value of bf16_encode(x): what a bfloat16 store of x holds."""
    return bf16_decode(bf16_encode(x))


# ----------------------------------------------------------- FP8 E4M3 (fn)

E4M3_EXP_BIAS = 7
E4M3_MAX = 448.0                    # S.1111.110 = 1.75 * 2**8
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUB_STEP_EXP = -9              # subnormal spacing 2**-6 / 2**3
E4M3_NAN = 0x7F


def e4m3_decode(codes):
    """uint8 E4M3 codes -> float64 values."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    f = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + f / 8.0, (e - E4M3_EXP_BIAS).astype(np.int32))
    sub = np.ldexp(f, E4M3_SUB_STEP_EXP)
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 0xF) & (f == 7), np.nan, val)
    return sign * val


def e4m3_encode_sat(x):
    """float values -> uint8 E4M3 codes: clamp to +-448, then round to nearest
    even on the E4M3 grid; the sign of zero is kept (-0 -> 0x80); NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    with np.errstate(invalid="ignore"):
        mant, ex = np.frexp(a)
        e = ex.astype(np.int64) - 1
        q = np.rint((2.0 * mant - 1.0) * 8.0)
        carry = q >= 8.0
        e = np.where(carry, e + 1, e)
        q = np.where(carry, 0.0, q)
        normal_code = ((e + E4M3_EXP_BIAS) << 3) | q.astype(np.int64)
        qs = np.rint(np.ldexp(a, -E4M3_SUB_STEP_EXP)).astype(np.int64)
        code = np.where(a < E4M3_MIN_NORMAL, qs, normal_code)
        code = np.where(np.isnan(x), E4M3_NAN, code | (sign << 7))
    return code.astype(np.uint8)


def e4m3_ordinal(codes):
    """Position of each finite code on the number line, +0 and -0 adjacent.

    Used to measure how many representable steps two codes lie apart."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    return np.where((c >> 7) & 1, -mag - 1, mag)
