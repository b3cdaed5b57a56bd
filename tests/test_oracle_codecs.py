"""Pins of the oracle's number formats against library routines and the formats'
definitions (no GPU)."""

import numpy as np
import pytest
import torch

from oracle import codecs as C


def _torch_bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_decode_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = C.bf16_bits_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_rne_against_torch_cast():
    # every upper half with low halves below, at and above the tie, plus random lows
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = [0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF]
    rng = np.random.default_rng(1)
    cases = [hi | l for l in lows] + [hi | rng.integers(0, 1 << 16, hi.size, dtype=np.uint32)]
    u = np.concatenate(cases).astype(np.uint32)
    x = u.view(np.float32)
    ours = C.f32_to_bf16_bits(x)
    ref = _torch_bf16_bits(x)
    fin = ~np.isnan(x)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.all((ours[~fin] & 0x7FFF) > 0x7F80)  # NaN stays NaN


def test_e4m3_decode_table():
    codes = np.arange(256, dtype=np.uint8)
    ours = C.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    # the definition's landmarks
    assert ours[0x7E] == 448.0 and np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[0x01] == 2.0 ** -9 and ours[0x07] == 7 * 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert ours[0x38] == 1.0 and ours[0xB8] == -1.0 and ours[0x80] == 0.0
    assert np.all(np.diff(ours[:0x7F]) > 0)  # monotone over the positive codes


def _fp8_probe_values():
    """Every representable value, every midpoint, one fp32 ulp either side of each,
    2^21 random fp32 patterns below 464 in magnitude and the subnormal range."""
    vals = C.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    mids = np.append(mids, 464.0 - 2.0 ** -20)
    pts = np.concatenate([vals, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(-np.inf))
    rng = np.random.default_rng(2)
    rnd = rng.integers(0, 0x43E80000, 1 << 21, dtype=np.uint32).view(np.float32)  # < 464
    sub = rng.uniform(0, 2.0 ** -6, 1 << 16).astype(np.float32)
    x = np.concatenate([pts, up, dn, rnd, sub]).astype(np.float32)
    x = x[np.abs(x) < 464]
    return np.concatenate([x, -x])


def test_e4m3_encode_against_torch_cast():
    x = _fp8_probe_values()
    ours = C.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, e.g. x={x[bad[:5]]} ours={ours[bad[:5]]} torch={ref[bad[:5]]}"


def test_e4m3_saturation_and_specials():
    x = np.array([448.0, 463.99, 464.0, 1e6, np.inf, -1e30, -np.inf, 0.0, -0.0, np.nan], np.float32)
    q = C.e4m3_encode(x)
    assert list(q[:7]) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert q[7] == 0x00 and q[8] == 0x80 and q[9] == 0x7F


def test_e4m3_roundtrip_error_bound():
    rng = np.random.default_rng(3)
    x = rng.uniform(-448, 448, 1 << 18).astype(np.float32)
    y = C.e4m3_decode(C.e4m3_encode(x))
    a = np.abs(x.astype(np.float64))
    normal = a >= 2.0 ** -6
    assert np.all(np.abs(y - x)[normal] <= 2.0 ** -4 * a[normal])  # half ulp, 3 mantissa bits
    assert np.all(np.abs(y - x)[~normal] <= 2.0 ** -10)  # half the subnormal step


@pytest.mark.parametrize("n", [1, 7, 256, 1000])
def test_int8_absmax_roundtrip(n):
    rng = np.random.default_rng(n)
    for _ in range(50):
        x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 2)).astype(np.float32)
        q, s = C.quant_int8_absmax(x)
        assert q.dtype == np.int8 and s.dtype == np.float32
        assert np.all(np.abs(q.astype(int)) <= 127)
        assert np.max(np.abs(q.astype(int))) == 127
        err = np.abs(C.dequant(q, s).astype(np.float64) - x)
        assert np.all(err <= s / 2 * (1 + 2.0 ** -20) + 2.0 ** -24 * np.abs(x))


@pytest.mark.parametrize("n", [1, 5, 256, 999])
def test_uint8_absmax_roundtrip(n):
    rng = np.random.default_rng(100 + n)
    for _ in range(50):
        x = (rng.standard_normal(n) ** 2 * 10.0 ** rng.uniform(-9, 1)).astype(np.float32)
        q, s = C.quant_uint8_absmax(x)
        assert q.dtype == np.uint8 and q.max() == 255
        err = np.abs(C.dequant(q, s).astype(np.float64) - x)
        assert np.all(err <= s / 2 * (1 + 2.0 ** -20) + 2.0 ** -24 * np.abs(x))


def test_absmax_all_zero_blocks():
    q, s = C.quant_int8_absmax(np.zeros(256, np.float32))
    assert s == 0 and not q.any()
    q, s = C.quant_uint8_absmax(np.zeros(3, np.float32))
    assert s == 0 and not q.any()


def test_int8_rint_is_half_even():
    # x / s lands exactly on k + 1/2 for these values: s = 1 when amax = 127
    x = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5], np.float32)
    q, s = C.quant_int8_absmax(x)
    assert s == 1.0
    assert list(q) == [127, 0, 2, 2, 0, -2, -2]


def test_tiny_blocks_take_the_division_or_zero_path():
    # reciprocal overflows: codes come from x / s and still span the range
    x = np.array([3e-38, -1.5e-38, 1e-39, 0.0], np.float32)
    s, r, mode = C.block_scale(np.max(np.abs(x)), 127)
    assert mode == 2 and not np.isfinite(r) and s > 0
    q, s2 = C.quant_int8_absmax(x)
    assert s2 == s and q[0] == 127 and abs(int(q[1]) + 64) <= 1 and q[3] == 0  # s is subnormal here
    # scale underflows to zero: zero codes, zero scale
    q, s3 = C.quant_uint8_absmax(np.array([1e-45, 0.0], np.float32))
    assert s3 == 0 and not q.any()
    # ordinary block: reciprocal path
    assert C.block_scale(np.float32(2.0), 127)[2] == 1


def _rn_f32_exact(q):
    """Nearest-even binary32 to the rational q (exact reference, slow)."""
    from fractions import Fraction

    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    k = a / quantum
    n = k.numerator // k.denominator
    rem = k - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return np.float32(sign * float(n * quantum))


def test_fma32_against_exact_rationals():
    from fractions import Fraction

    rng = np.random.default_rng(12)
    a = (rng.standard_normal(6000) * 10.0 ** rng.integers(-8, 8, 6000)).astype(np.float32)
    b = (rng.standard_normal(6000) * 10.0 ** rng.integers(-8, 8, 6000)).astype(np.float32)
    c = (rng.standard_normal(6000) * 10.0 ** rng.integers(-8, 8, 6000)).astype(np.float32)
    # heavy cancellation: c close to -a*b
    c[:2000] = (-(a[:2000].astype(np.float64) * b[:2000]) * (1 + rng.standard_normal(2000) * 1e-7)).astype(np.float32)
    got = C.fma32(a, b, c)
    for i in range(a.size):
        want = _rn_f32_exact(Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i])))
        assert got[i].view(np.uint32) == want.view(np.uint32), (a[i], b[i], c[i], got[i], want)


def test_fma32_double_rounding_case():
    """a*b + c = 1 + 2^-23 + 2^-24 - 2^-70: just below the midpoint between
    1 + 2^-23 and 1 + 2^-22, so the answer is 1 + 2^-23; rounding to fp64 first
    would land on the midpoint and round to even (1 + 2^-22)."""
    a = np.float32(1 + 2.0 ** -23)
    b = np.float32(2.0 ** -24 * (1 - 2.0 ** -23))
    c = np.float32(1 + 2.0 ** -23)
    assert C.fma32(a, b, c) == np.float32(1 + 2.0 ** -23)
    assert np.float32(np.float64(a) * np.float64(b) + np.float64(c)) == np.float32(1 + 2.0 ** -22)
    assert C.fma32(-a, b, -c) == -np.float32(1 + 2.0 ** -23)


def test_fma32_without_addend_is_the_rounded_product():
    rng = np.random.default_rng(13)
    a = rng.standard_normal(100000).astype(np.float32)
    b = rng.standard_normal(100000).astype(np.float32)
    assert np.array_equal(C.fma32(a, b, np.zeros_like(a)).view(np.uint32), (a * b).view(np.uint32))
