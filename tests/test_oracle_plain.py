"""Pins of the oracle's two arithmetic legs against exact rational arithmetic.

The pages fix the method (Adam with block-quantised state, block-wise FP8 of the
updated parameters) but no order of fp32 operations.  The oracle carries two
restatements: the contract leg (oracle.adam8 / oracle.fp8 / oracle.codecs: fused
multiply-adds, reciprocal bias corrections, codes from the product with a
reciprocal block scale) that the kernels reproduce bit for bit, and the plain leg
(oracle.plain: every operation separate, division by the bias corrections and by
the block scale).  Here each leg is recomputed element by element with Python's
exact rationals, rounding to the nearest fp32 (ties to even) only where its
stated form rounds; the inputs include rounding ties and elements on which the
two forms give different results, so swapping one form for the other anywhere
in either leg fails a test."""

from fractions import Fraction as Q

import numpy as np
import pytest

from oracle import adam8 as OA
from oracle import codecs as OC
from oracle import fp8 as OF
from oracle import plain as PL

F32 = np.float32


# ----------------------------------------------------------------------------- exact rounding


def _binade(a):
    """e with 2^e <= a < 2^(e+1) for a rational a > 0."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Q(2) ** e > a:
        e -= 1
    while Q(2) ** (e + 1) <= a:
        e += 1
    return e


def rint_he(x):
    """The integer nearest the rational x, ties to even."""
    fl = x.numerator // x.denominator
    rem = x - fl
    if rem > Q(1, 2) or (rem == Q(1, 2) and fl % 2):
        fl += 1
    return fl


def rnd32(x):
    """The fp32 number nearest the rational x (ties to even, subnormals,
    overflow to infinity)."""
    if x == 0:
        return F32(0.0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = max(_binade(a), -126)
    quantum = Q(2) ** (e - 23)
    val = rint_he(a / quantum) * quantum
    if val >= Q(2) ** 128:
        return F32(sign * np.inf)
    return F32(sign * float(val))


def q(x):
    return Q(float(F32(x)))


def sqrt32(x):
    """Correctly rounded fp32 square root of the fp32 x >= 0: the candidate whose
    rounding interval [mid-, mid+] holds sqrt(x), decided on exact squares."""
    x = F32(x)
    if x == 0:
        return F32(0.0)
    c = F32(np.sqrt(np.float64(x)))
    for y in (c, np.nextafter(c, F32(np.inf)), np.nextafter(c, F32(0))):
        lo = (q(np.nextafter(y, F32(0))) + q(y)) / 2
        hi = (q(y) + q(np.nextafter(y, F32(np.inf)))) / 2
        if lo * lo <= q(x) <= hi * hi:
            return F32(y)
    raise AssertionError("no candidate")


def e4m3_round(x):
    """x rounded to the E4M3 grid (binade quantum 2^(e-3), subnormal step 2^-9,
    ties to even, saturating at +-448), as a rational."""
    if x == 0:
        return Q(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = max(_binade(a), -6)
    quantum = Q(2) ** (e - 3)
    val = rint_he(a / quantum) * quantum
    return sign * min(val, Q(448))


# ----------------------------------------------------------------------------- exact restatements of the two legs


def adam_exact(g, p, m, v, hp, plain):
    """One element of the Adam update in exact rationals, rounded where the leg
    rounds.  g, p, m, v: fp32; hp: that leg's hyper-parameters."""
    g, p, m, v = q(g), q(p), q(m), q(v)
    H = {k: q(x) for k, x in hp.items()}
    gg = rnd32(g * g)
    if plain:
        m1 = rnd32(q(rnd32(H["b1"] * m)) + q(rnd32(H["omb1"] * g)))
        v1 = rnd32(q(rnd32(H["b2"] * v)) + q(rnd32(H["omb2"] * q(gg))))
        mh = rnd32(q(m1) / H["bc1"])
        vh = rnd32(q(v1) / H["bc2"])
    else:  # fused multiply-adds: the product enters the sum exactly
        m1 = rnd32(H["b1"] * m + q(rnd32(H["omb1"] * g)))
        v1 = rnd32(H["b2"] * v + q(rnd32(H["omb2"] * q(gg))))
        mh = rnd32(q(m1) * H["rbc1"])
        vh = rnd32(q(v1) * H["rbc2"])
    den = rnd32(q(sqrt32(vh)) + H["eps"])
    u = rnd32(q(mh) / q(den))
    if plain:
        p1 = rnd32(p - q(rnd32(H["lr"] * q(u))))
    else:
        p1 = rnd32(p - H["lr"] * q(u))
    return p1, m1, v1


def quant_exact(x, qmax, lo, hi, plain):
    """Codes and scale of one block in exact rationals."""
    xs = [q(a) for a in x]
    amax = max(abs(a) for a in xs) if lo < 0 else max(xs)
    s = rnd32(amax / qmax)
    if s == 0:
        return [0] * len(xs), F32(0)
    r = rnd32(Q(qmax) / amax)
    if plain or not np.isfinite(r):
        codes = [rint_he(q(rnd32(a / q(s)))) for a in xs]
    else:
        codes = [rint_he(a * q(r)) for a in xs]
    return [min(max(c, lo), hi) for c in codes], s


def fp8_exact(p, plain):
    """E4M3 values (rational) and scale of one tile in exact rationals."""
    ps = [q(a) for a in p]
    amax = max(abs(a) for a in ps)
    s = rnd32(amax / 448)
    if s == 0:
        return None, F32(0)
    r = rnd32(Q(448) / amax)
    if plain or not np.isfinite(r):
        vals = [e4m3_round(q(rnd32(a / q(s)))) for a in ps]
    else:
        vals = [e4m3_round(q(rnd32(a * q(r)))) for a in ps]
    return vals, s


# ----------------------------------------------------------------------------- the rounding helpers themselves


def test_exact_helpers_against_hardware_fp32():
    """rnd32 / sqrt32 agree with numpy's fp32 arithmetic on exact products and
    quotients (numpy's fp32 ops are single IEEE roundings)."""
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(300) * 10.0 ** rng.integers(-30, 30, 300)).astype(np.float32)
    b = (rng.standard_normal(300) * 10.0 ** rng.integers(-5, 5, 300)).astype(np.float32)
    for x, y in zip(a, b):
        assert rnd32(q(x) * q(y)) == x * y
        assert rnd32(q(x) / q(y)) == x / y
        assert rnd32(q(x) + q(y)) == x + y
        assert sqrt32(abs(x)) == np.sqrt(abs(x))
    assert rnd32(Q(1) + Q(1, 2 ** 24)) == F32(1.0)  # tie to even
    assert rnd32(Q(1) + Q(3, 2 ** 24)) == F32(1.0) + F32(2.0 ** -22)  # tie to even, upward
    assert rnd32(Q(1, 2 ** 150)) == 0 and rnd32(Q(3, 2 ** 151)) == F32(2.0 ** -149)
    assert rint_he(Q(5, 2)) == 2 and rint_he(Q(7, 2)) == 4 and rint_he(Q(-5, 2)) == -2


# ----------------------------------------------------------------------------- Adam update


def _adam_inputs(n, seed):
    rng = np.random.default_rng(seed)
    g = OC.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = (rng.standard_normal(n) * 1e-3).astype(np.float32) ** 2
    return g, p, m, v


@pytest.mark.parametrize("t", [1, 10, 1000])
def test_both_adam_legs_exact(t):
    g, p, m, v = _adam_inputs(400, t)
    hc = OA.adam_hparams(1e-3, 0.9, 0.999, 1e-8, t)
    hpl = PL.adam_hparams(1e-3, 0.9, 0.999, 1e-8, t)
    pc, mc, vc = OA.adam_update(g, p, m, v, hc)
    pp, mp, vp = PL.adam_update(g, p, m, v, hpl)
    gf = OC.bf16_bits_to_f32(g)
    differ = dict(m=0, v=0, p=0)
    for k in range(len(p)):
        want_c = adam_exact(gf[k], p[k], m[k], v[k], hc, plain=False)
        want_p = adam_exact(gf[k], p[k], m[k], v[k], hpl, plain=True)
        assert (pc[k], mc[k], vc[k]) == want_c, (k, "contract")
        assert (pp[k], mp[k], vp[k]) == want_p, (k, "plain")
        differ["p"] += want_c[0] != want_p[0]
        differ["m"] += want_c[1] != want_p[1]
        differ["v"] += want_c[2] != want_p[2]
    # the two forms really differ on these inputs: a swap of one for the other
    # in either leg cannot pass the element checks above
    assert differ["m"] > 0 and differ["v"] > 0 and differ["p"] > 0, differ


def test_plain_adam_hparams_are_bias_corrections():
    h = PL.adam_hparams(1e-3, 0.9, 0.999, 1e-8, 10)
    assert h["bc1"] == F32(1 - 0.9 ** 10) and h["bc2"] == F32(1 - 0.999 ** 10)
    assert h["omb1"] == F32(1 - 0.9) and h["omb2"] == F32(1 - 0.999)


# ----------------------------------------------------------------------------- block quantisers


def _blocks(seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(60):
        out.append((rng.standard_normal(256) * 10.0 ** rng.uniform(-6, 1)).astype(np.float32))
    # ties: a power-of-two scale (amax = 127 * 2^-10) and codes at k + 1/2
    tie = np.array([127, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -126.5], np.float32) * np.float32(2.0 ** -10)
    out.append(tie)
    # near ties: elements at (k + 1/2) * s for a scale s that is not a power of
    # two, where x*r and fp32(x/s) straddle the midpoint in both directions
    for amax in (rng.uniform(0.5, 1.0, 6) * 10.0 ** rng.uniform(-6, 0, 6)).astype(np.float32):
        s = amax / F32(127)
        ks = np.arange(-126, 127, dtype=np.float32)
        out.append(np.concatenate([[amax], ((ks + F32(0.5)) * s).astype(np.float32)]).astype(np.float32))
    out.append(np.zeros(16, np.float32))  # all zero: zero scale, zero codes
    out.append(np.array([3e-45, -1e-45, 0.0], np.float32))  # scale underflows to 0: zero codes
    out.append(np.array([2e-38, -1e-38, 5e-39], np.float32))  # reciprocal overflows: codes from x / s
    return out


def test_int8_quantiser_legs_exact():
    differ = 0
    for x in _blocks(7):
        qc, sc = OC.quant_int8_absmax(x)
        qp, sp = PL.quant_int8(x)
        cc, s1 = quant_exact(x, 127, -127, 127, plain=False)
        cp, s2 = quant_exact(x, 127, -127, 127, plain=True)
        assert sc == s1 and sp == s2
        assert qc.tolist() == cc and qp.tolist() == cp
        differ += int(np.sum(qc != qp))
    assert differ > 0  # x*r and x/s disagree somewhere: a swap fails


def test_uint8_quantiser_legs_exact():
    differ = 0
    rng = np.random.default_rng(11)
    near = []
    for amax in (rng.uniform(0.5, 1.0, 6) * 10.0 ** rng.uniform(-9, -3, 6)).astype(np.float32):
        s = amax / F32(255)
        ks = np.arange(0, 255, dtype=np.float32)
        near.append(np.concatenate([[amax], ((ks + F32(0.5)) * s).astype(np.float32)]).astype(np.float32))
    for x in _blocks(8) + near:
        x = np.abs(x)
        qc, sc = OC.quant_uint8_absmax(x)
        qp, sp = PL.quant_uint8(x)
        cc, s1 = quant_exact(x, 255, 0, 255, plain=False)
        cp, s2 = quant_exact(x, 255, 0, 255, plain=True)
        assert sc == s1 and sp == s2
        assert qc.tolist() == cc and qp.tolist() == cp
        differ += int(np.sum(qc != qp))
    assert differ > 0


def test_quantiser_ties_go_to_even():
    x = np.array([127, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -126.5], np.float32) * np.float32(2.0 ** -10)
    for quant in (OC.quant_int8_absmax, PL.quant_int8):
        codes, s = quant(x)
        assert s == F32(2.0 ** -10)
        assert codes.tolist() == [127, 2, 4, -2, 0, 0, 2, -126]


# ----------------------------------------------------------------------------- FP8 tiles


def _tiles(seed):
    rng = np.random.default_rng(seed)
    out = [(rng.standard_normal(128) * 10.0 ** rng.uniform(-4, 0)).astype(np.float32) for _ in range(80)]
    # near ties: elements at midpoints of the E4M3 grid times s
    grid = OC.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    for amax in (rng.uniform(0.5, 1.0, 6) * 10.0 ** rng.uniform(-4, 0, 6)).astype(np.float32):
        s = amax / F32(448)
        out.append(np.concatenate([[amax], (mids * s).astype(np.float32), (-mids * s).astype(np.float32)]))
    out.append(np.array([1e-37, -3e-38, 4e-39], np.float32))  # reciprocal overflows
    out.append(np.array([5e-43, -2e-44], np.float32))  # scale underflows: signed zero codes
    return out


def test_fp8_legs_exact():
    differ = 0
    for p in _tiles(9):
        for leg, plain in ((OF.fp8_tile, False), (PL.fp8_tile, True)):
            codes, s = leg(p)
            vals, s_want = fp8_exact(p, plain)
            assert s == s_want
            if vals is None:
                assert codes.tolist() == [0x80 if np.signbit(a) else 0 for a in p]
                continue
            got = OC.e4m3_decode(codes)
            assert [Q(float(a)) for a in got] == vals, plain
        differ += int(np.sum(OF.fp8_tile(p)[0] != PL.fp8_tile(p)[0]))
    assert differ > 0
