"""Oracle encoders: float64 values -> storage codes of the cache element types.

Test infrastructure only (see oracle/__init__.py). Every encoder here is a
single rounding from float64, written from the format definitions:

* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits; normals from
  2**-126, subnormal step 2**-133, largest finite (2 - 2**-7) * 2**127.
  Round to nearest, ties to even; magnitudes that round past the largest
  finite value become infinity (IEEE behaviour).
* float16 (IEEE binary16): numpy's float64 -> float16 conversion, which is a
  single round-to-nearest-even (a library routine, allowed as a step).
* FP8 E4M3FN (OCP 8-bit floating point, "FN" = finite + NaN only):
  1-4-3, bias 7, no infinities, S.1111.111 is NaN, largest finite
  1.75 * 2**8 = 448, normals from 2**-6, subnormal step 2**-9.
* FP8 E5M2 (OCP): 1-5-2, bias 15, largest finite 1.75 * 2**15 = 57344,
  normals from 2**-14, subnormal step 2**-16.
  Both FP8 encoders saturate: a finite magnitude beyond the largest finite
  value encodes as that value ("satfinite"), i.e. the code of
  round-to-nearest-even(saturate(v)). The aclnnKvRmsNormRopeCache page
  ("Restrictions on quantization scenarios") names the formats but no
  rounding rule; saturating RNE is the reading taken.
* int8: round half to even, then clamp to [-128, 127].

Codes are returned as unsigned integer arrays (uint16 for 16-bit types,
uint8 for 8-bit types) so that caches can be compared bit for bit.
"""
import numpy as np

DTYPES_16 = ("bf16", "f16")
DTYPES_8 = ("int8", "fp8_e4m3fn", "fp8_e5m2")


def _round_to_grid(a, man_bits, emin):
    """Round |values| a >= 0 (float64) to the nearest point of a binary
    floating-point grid with `man_bits` fraction bits and smallest normal
    exponent `emin`; ties go to the even grid point. Exact in float64 for
    every grid used here (all scalings are by powers of two)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    nz = a > 0
    _, E = np.frexp(a[nz])                 # a = m * 2**E, m in [0.5, 1)
    e = np.maximum(E - 1, emin)            # binade exponent, clamped at the subnormal range
    ulp = np.ldexp(1.0, e - man_bits)
    out[nz] = np.rint(a[nz] / ulp) * ulp   # np.rint: round half to even
    return out


def bf16_encode(v):
    """float64 -> bfloat16 bit patterns (uint16), one RNE rounding."""
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v)
    q = _round_to_grid(np.abs(np.where(np.isnan(v), 0.0, v)), 7, -126)
    q = np.where(q >= 2.0 ** 128, np.inf, q)
    q = np.where(np.isinf(v), np.inf, q)
    bits = (np.abs(q).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(np.isnan(v), np.uint16(0x7FC0), bits)
    return (bits | (sign.astype(np.uint16) << 15)).astype(np.uint16)


def bf16_decode(bits):
    """bfloat16 bit patterns -> float64 values (exact)."""
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f16_encode(v):
    """float64 -> IEEE binary16 bit patterns (uint16), numpy's single RNE rounding."""
    with np.errstate(over="ignore", invalid="ignore"):
        return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


def f16_decode(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _fp8_encode(v, man_bits, bias, emin, maxfinite, nan_code):
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v).astype(np.uint8) << 7
    a = np.minimum(np.abs(np.where(np.isnan(v), 0.0, v)), maxfinite)   # saturate first
    q = np.minimum(_round_to_grid(a, man_bits, emin), maxfinite)
    code = np.zeros(q.shape, dtype=np.int64)
    nz = q > 0
    _, E = np.frexp(q[nz])
    e = E - 1
    sub = e < emin
    qn = q[nz]
    c = np.where(
        sub,
        np.rint(qn / 2.0 ** (emin - man_bits)),                                 # exponent field 0
        ((e + bias) << man_bits) + np.rint(qn / np.ldexp(1.0, e) * 2 ** man_bits) - 2 ** man_bits,
    )
    code[nz] = c.astype(np.int64)
    code = code.astype(np.uint8) | sign
    return np.where(np.isnan(v), np.uint8(nan_code) | sign, code).astype(np.uint8)


def fp8_e4m3fn_encode(v):
    """float64 -> OCP FP8 E4M3FN codes (uint8), saturating RNE."""
    return _fp8_encode(v, 3, 7, -6, 448.0, 0x7F)


def fp8_e5m2_encode(v):
    """float64 -> OCP FP8 E5M2 codes (uint8), saturating RNE."""
    return _fp8_encode(v, 2, 15, -14, 57344.0, 0x7F)


def _fp8_decode(codes, man_bits, bias, emin):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> man_bits) & ((0x7F >> man_bits))
    m = c & ((1 << man_bits) - 1)
    val = np.where(ef == 0,
                   m * 2.0 ** (emin - man_bits),
                   (1.0 + m / 2 ** man_bits) * np.ldexp(1.0, (ef - bias)))
    return s * val


def fp8_e4m3fn_decode(codes):
    """E4M3FN codes -> float64 (the NaN codes 0x7F/0xFF decode as NaN)."""
    c = np.asarray(codes, dtype=np.uint8)
    out = _fp8_decode(c, 3, 7, -6)
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def fp8_e5m2_decode(codes):
    """E5M2 codes -> float64 (exponent field 31: infinities and NaNs)."""
    c = np.asarray(codes, dtype=np.uint8)
    out = _fp8_decode(c, 2, 15, -14)
    inf = (c & 0x7C) == 0x7C
    out = np.where(inf & ((c & 0x3) == 0), np.where(c & 0x80, -np.inf, np.inf), out)
    return np.where(inf & ((c & 0x3) != 0), np.nan, out)


def int8_encode(v):
    """float64 -> int8 codes (returned as uint8 bit patterns): RNE, clamp [-128, 127]."""
    q = np.clip(np.rint(np.asarray(v, dtype=np.float64)), -128, 127).astype(np.int8)
    return q.view(np.uint8)


def int8_decode(codes):
    return np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.float64)


def encode(v, dtype):
    """Dispatch on the cache element type name."""
    return {
        "bf16": bf16_encode,
        "f16": f16_encode,
        "int8": int8_encode,
        "fp8_e4m3fn": fp8_e4m3fn_encode,
        "fp8_e5m2": fp8_e5m2_encode,
    }[dtype](v)


def decode(codes, dtype):
    return {
        "bf16": bf16_decode,
        "f16": f16_decode,
        "int8": int8_decode,
        "fp8_e4m3fn": fp8_e4m3fn_decode,
        "fp8_e5m2": fp8_e5m2_decode,
    }[dtype](codes)


def code_dtype(dtype):
    """numpy container type of one code."""
    return np.uint16 if dtype in DTYPES_16 else np.uint8


def code_ordinal(codes, dtype):
    """Position of each code on the ordered code line (monotone in the encoded
    value, +0 and -0 share position 0), used for 'within one code' checks."""
    c = np.asarray(codes).astype(np.int64)
    if dtype == "int8":
        return np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.int64)
    if dtype in DTYPES_16:
        mag = c & 0x7FFF
        return np.where(c & 0x8000, -mag, mag)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)
