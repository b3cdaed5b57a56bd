"""Number formats used on the DBuffer step (oracle; test infrastructure only).

* bf16: gradients are bf16 in and out of the fused pre-communication op
  ("veScale-FSDP: Flexible and High-Performance FSDP at Scale", Method: the
  group-level add / scale / zero / copy).  Rounding is IEEE round-to-nearest-even.
* FP8 E4M3: block-wise FP8 parameters "DeepSeek-V3 style" (same page, TL;DR and
  Key claims).  The pages do not define the format; this is the OCP 8-bit
  floating point E4M3 encoding (bias 7, 3 mantissa bits, no infinities, the single
  NaN pattern S.1111.111, largest finite 448, subnormal step 2^-9), written here
  from that definition, with round-to-nearest-even and saturation to +-448.
* int8 / uint8 linear absmax block quantisers for the 8-bit Adam state ("8-bit
  Adam" in Key claims; the pages give block locality but no quantiser, so the
  reading is a symmetric linear map with one fp32 absmax scale per block; codes
  are the product with the reciprocal scale, computed once per block, rounded
  once to an integer).
* fma32: the fp32 fused multiply-add (one rounding), used by the Adam update.

Everything is numpy; fp32 arithmetic is done on float32 arrays so that every
operation is one IEEE fp32 operation rounded to nearest.
"""

import numpy as np

F32 = np.float32

# ----------------------------------------------------------------------------- bf16


def f32_to_bf16_bits(x):
    """fp32 -> bf16 bit pattern (uint16), round to nearest, ties to even.

    The 16 low bits are dropped after adding half an ulp of the kept part, with the
    tie going to the even kept mantissa; NaNs stay (quiet) NaNs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    is_nan = (u & 0x7FFFFFFF) > 0x7F800000
    keep_lsb = (u >> 16) & 1
    rounded = (u + 0x7FFF + keep_lsb) >> 16
    quiet = (u >> 16) | 0x40
    return np.where(is_nan, quiet, rounded).astype(np.uint16)


def bf16_bits_to_f32(b):
    """bf16 bit pattern -> the fp32 value it denotes (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- fused multiply-add


def fma32(a, b, c):
    """fp32 fused multiply-add: a*b + c rounded once to nearest-even fp32.

    The product of two fp32 numbers is exact in fp64; the fp64 sum s = a*b + c
    is corrected by its exact error e (Knuth's TwoSum: s + e == a*b + c).  The
    fp64 rounding of s can only matter when s falls exactly on a midpoint between
    two fp32 numbers: any other s lies at least one fp64 ulp from every fp32
    midpoint while |e| is at most half an fp64 ulp.  At such a midpoint the sign
    of e decides (e == 0 is a true tie: nearest even)."""
    a64 = np.asarray(a, np.float32).astype(np.float64)
    b64 = np.asarray(b, np.float32).astype(np.float64)
    c64 = np.asarray(c, np.float32).astype(np.float64)
    p = a64 * b64
    s = p + c64
    bp = s - p
    e = (p - (s - bp)) + (c64 - bp)
    with np.errstate(over="ignore", invalid="ignore"):
        r = s.astype(np.float32)
        r64 = r.astype(np.float64)
        up = np.nextafter(r, np.float32(np.inf))
        dn = np.nextafter(r, np.float32(-np.inf))
        lo = np.where(r64 < s, r, dn)
        hi = np.where(r64 < s, up, r)
        mid = (lo.astype(np.float64) + hi.astype(np.float64)) / 2 == s
    tie_break = mid & (r64 != s) & (e != 0)
    return np.where(tie_break, np.where(e > 0, hi, lo), r).astype(np.float32)


# ----------------------------------------------------------------------------- FP8 E4M3

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def e4m3_decode(codes):
    """FP8 E4M3 code (uint8) -> float64 value, from the format's definition.

    exponent field E (4 bits, bias 7), mantissa M (3 bits):
    E == 0        -> subnormal  M * 2^-9
    E == 15, M==7 -> NaN
    otherwise     -> 2^(E-7) * (1 + M/8)
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m * 2.0 ** -9
    nrm = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int32))
    val = np.where(e == 0, sub, nrm)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def e4m3_encode(x):
    """fp32 -> FP8 E4M3 code (uint8): round to nearest even, saturate to +-448.

    |x| >= 448 (and +-inf) -> +-448 (the "satfinite" rule); NaN -> 0x7F.  For
    |x| < 448 the result is the nearest multiple of the quantum at |x|'s binade,
    2^(e-3) with e = max(floor(log2|x|), -6) (below 2^-6 the quantum is the
    subnormal step 2^-9), ties to the even multiple.  The sign of zero is kept."""
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    bits = x32.view(np.uint32)
    neg = (bits >> 31).astype(np.uint8)
    a = np.abs(x32.astype(np.float64))  # exact
    is_nan = np.isnan(a)
    sat = (a >= E4M3_MAX) & ~is_nan

    safe = np.where((a > 0) & ~sat & ~is_nan, a, 1.0)
    _, ex = np.frexp(safe)  # safe = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)  # floor(log2 a), clamped to the lowest normal binade
    quantum = np.ldexp(1.0, (e - 3).astype(np.int32))
    r = np.rint(safe / quantum)  # exact quotient, half-to-even
    val = r * quantum  # representable by construction (r <= 16 within the binade)
    val = np.where(a > 0, val, 0.0)

    # encode the (exact) representable value
    is_sub = val < 2.0 ** -6
    m_sub = np.rint(val / 2.0 ** -9).astype(np.int64)
    vs = np.where(val > 0, val, 1.0)
    _, ex2 = np.frexp(vs)
    E = (ex2 - 1) + 7
    M = np.rint((vs / np.ldexp(1.0, (ex2 - 1).astype(np.int32)) - 1.0) * 8.0).astype(np.int64)
    code = np.where(is_sub, m_sub, (E << 3) | M)
    code = np.where(sat, 0x7E, code)
    code = np.where(is_nan, E4M3_NAN, code | (neg.astype(np.int64) << 7))
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------- linear absmax block quantisers


def block_scale(amax, qmax):
    """(stored scale s, reciprocal r, mode) of a block with absmax amax mapped to
    qmax.  s = amax / qmax and r = qmax / amax, each one fp32 division.
    mode 0: s == 0 (all-zero block, or amax so small that s underflows): codes 0;
    mode 1: r finite: codes from x * r;
    mode 2: r overflowed (amax below ~qmax / 3.4e38): codes from x / s."""
    with np.errstate(over="ignore", divide="ignore"):
        s = F32(amax) / F32(qmax)
        r = F32(qmax) / F32(amax)
    if s == 0:
        return F32(0), r, 0
    return F32(s), r, (1 if np.isfinite(r) else 2)


def scaled(x, s, r, mode):
    """x * r (mode 1) or x / s (mode 2), fp32."""
    x = np.asarray(x, dtype=np.float32)
    return x * r if mode == 1 else x / s


def rint_product(x, r):
    """rint of the exact product x*r (fp32 x, fp32 r), ties to even: the fp64
    product is exact and fp64 rint is exact."""
    return np.rint(np.asarray(x, np.float32).astype(np.float64) * np.float64(np.float32(r)))


def quant_int8_absmax(x):
    """One block of signed state -> (int8 codes, fp32 scale).

    s = max|x| / 127 is the stored scale; with the reciprocal r = 127 / max|x|
    (one fp32 division per block) code = clamp(rint(x * r), -127, 127) where the
    product is rounded once, directly to an integer (half to even); when r
    overflows, code = clamp(rint(fp32(x / s))).  A block whose scale is 0 gets
    zero codes; -128 is never produced."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.max(np.abs(x)) if x.size else F32(0)
    s, r, mode = block_scale(amax, 127)
    if mode == 0:
        return np.zeros(x.shape, np.int8), F32(0)
    y = rint_product(x, r) if mode == 1 else np.rint(x / s)
    return np.clip(y, -127, 127).astype(np.int8), s


def quant_uint8_absmax(x):
    """One block of non-negative state -> (uint8 codes, fp32 scale).

    s = max x / 255; code = clamp(rint(x * r), 0, 255) with r = 255 / max x and
    the product rounded once to an integer (x / s when r overflows); a block
    whose scale is 0 gets zero codes."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.max(x) if x.size else F32(0)
    s, r, mode = block_scale(amax, 255)
    if mode == 0:
        return np.zeros(x.shape, np.uint8), F32(0)
    y = rint_product(x, r) if mode == 1 else np.rint(x / s)
    return np.clip(y, 0, 255).astype(np.uint8), s


def dequant(codes, scale):
    """code * scale, one fp32 multiplication per element."""
    return np.asarray(codes).astype(np.float32) * F32(scale)
