"""Every branch of the block quantisers on the GPU, against the oracle bit for bit.

A block's stored scale is s = amax / qmax and its codes come from the product
with r = qmax / amax; two branches leave that path:
  * r overflows (amax below about qmax / 3.4e38): codes from x / s;
  * s underflows to 0 although amax is not 0: zero codes (as for an all-zero
    block).
The same holds for the FP8 tiles (qmax = 448: r overflows below about 1.3e-36,
s underflows below about 3.1e-43).  The seeded workloads never reach these
magnitudes, so here whole tensors (and, in the mixed tensors, individual Adam
blocks) are given states that drive each Adam kernel family (flat 256 / 128 / 32
blocks, 256-column strips, bands of tensors with C % 256 != 0, 128x128 and 32x32
tiles) and each FP8 path (fused and standalone) into every branch:
  TINY_M   gradient 0, m = code * 2e-39 (subnormal scale): m' amax ~ 2e-37, r_m
           overflows; v normal; master ~ N(0, 1e-37): the FP8 tile's r overflows
  TINY_V   gradient 0, m = 0, v = code * 2e-39: r_v overflows; master tiny
  UNDER    gradient 0, m = code * 2^-149 with |code| <= 70, v = code * 2^-149
           with code <= 127: both scales underflow to 0 (zero codes)
  UNDER8   gradient 0, m = 0, master = k * 2^-149 with |k| <= 200: the FP8
           scale underflows to 0 (codes +-0 by sign)
  NORMAL   the seeded workload's distributions
"""

import numpy as np
import pytest

import workloads as W
from _step_harness import StepCase
from oracle import adam8 as OA
from oracle import codecs as OC
from oracle import fp8 as OF
from oracle import planner as P
from test_parity_step import _compare

pytestmark = pytest.mark.gpu

NORMAL, TINY_M, TINY_V, UNDER, UNDER8, MIXED = range(6)


def _tensors():
    T = W.TensorSpec
    return [
        (T("tiny_1d", 1, 1000, 256, W.ADAM_FLAT256, True), TINY_M),
        (T("under_1d", 1, 600, 256, W.ADAM_FLAT256, True), UNDER),
        (T("tiny_strip", 128, 256, 128 * 256, W.ADAM_FLAT256, True), TINY_M),
        (T("under8_strip", 130, 512, 128 * 512, W.ADAM_FLAT256, True), UNDER8),
        (T("tinyv_band", 200, 360, 128 * 360, W.ADAM_FLAT256, True), TINY_V),
        (T("mixed_band", 140, 360, 128 * 360, W.ADAM_FLAT256, True), MIXED),
        (T("tiny_tile", 140, 200, 128 * 200, W.ADAM_TILE128, True), TINY_M),
        (T("under8_tile", 129, 136, 128 * 136, W.ADAM_TILE128, True), UNDER8),
        (T("mixed_tile_1d", 1, 300, 128, W.ADAM_TILE128, True), MIXED),
        (T("mixed_tile", 256, 384, 128 * 384, W.ADAM_TILE128, True), MIXED),
        (T("mixed_t32", 70, 40, 32 * 40, W.ADAM_TILE32, False), MIXED),
        (T("mixed_strip", 256, 512, 128 * 512, W.ADAM_FLAT256, True), MIXED),
        (T("normal_strip", 128, 512, 128 * 512, W.ADAM_FLAT256, True), NORMAL),
    ]


def _craft(case, regimes, seed):
    """Overwrite the case's inputs block by block with the regimes' states."""
    rng = np.random.default_rng(seed)
    L, lo, hi, S = case.olayout, case.dev_lo, case.dev_hi, case.S
    n = case.n
    tensor_of = np.full(n, -1, np.int64)
    toff_of = np.zeros(n, np.int64)
    for k, i, t_off, ln, loff, _, _ in L.intervals[L.dev_table[lo][0]:L.dev_table[hi][0]]:
        p0 = (k - lo) * S + loff
        tensor_of[p0:p0 + ln] = i
        toff_of[p0:p0 + ln] = np.arange(t_off, t_off + ln)
    used = set()
    for slot, pos in P.adam_blocks(L, lo, hi):
        i = int(tensor_of[pos[0]])
        reg = regimes[i] if regimes[i] != MIXED else int(slot) % 5
        used.add(reg)
        if reg == NORMAL:
            continue
        bits, base = case.grads[i]
        bits[toff_of[pos] - base] = 0  # gradient 0
        k = len(pos)
        if reg == TINY_M:
            case.m[pos] = rng.integers(-127, 128, k)
            case.ms[slot] = np.float32(2e-39)
            case.v[pos] = rng.integers(64, 256, k)
            case.vs[slot] = np.float32(1e-6 / 255)
            case.master[pos] = (rng.standard_normal(k) * 1e-37).astype(np.float32)
        elif reg == TINY_V:
            case.m[pos] = 0
            case.ms[slot] = np.float32(1e-5)
            case.v[pos] = rng.integers(64, 256, k)
            case.vs[slot] = np.float32(2e-39)
            case.master[pos] = (rng.standard_normal(k) * 1e-37).astype(np.float32)
        elif reg == UNDER:
            case.m[pos] = rng.integers(-70, 71, k)
            case.ms[slot] = np.float32(2.0 ** -149)
            case.v[pos] = rng.integers(0, 128, k)
            case.vs[slot] = np.float32(2.0 ** -149)
        elif reg == UNDER8:
            case.m[pos] = 0
            case.ms[slot] = np.float32(1e-5)
            case.master[pos] = rng.integers(-200, 201, k).astype(np.float32) * np.float32(2.0 ** -149)
    return used


def _modes(case):
    """Quantiser branch taken by every m / v block and FP8 tile, per the oracle:
    'zero' (amax 0), 'underflow' (amax > 0, scale 0), 'recip' (codes from x*r),
    'div' (r overflowed)."""
    L, lo, hi = case.olayout, case.dev_lo, case.dev_hi
    want = case.run_oracle()

    def mode(amax, qmax):
        s, r, md = OC.block_scale(amax, qmax)
        return "zero" if amax == 0 else ("underflow", "recip", "div")[md]

    dbuf = want["dbuf"]
    seen = {"m": set(), "v": set(), "fp8": set()}
    for slot, pos in P.adam_blocks(L, lo, hi):
        m = OC.dequant(case.m[pos], case.ms[slot])
        v = OC.dequant(case.v[pos], case.vs[slot])
        _, m1, v1 = OA.adam_update(dbuf[pos], case.master[pos], m, v, case.hp_o)
        seen["m"].add(mode(np.max(np.abs(m1)), 127))
        seen["v"].add(mode(np.max(v1), 255))
    for slot, pos in P.fp8_tiles(L, lo, hi):
        seen["fp8"].add(mode(np.max(np.abs(want["master"][pos])), 448))
    return want, seen


@pytest.mark.parametrize("dev", [(0, 1), (0, 3), (1, 3)])
def test_quantiser_branches_match_oracle(cuda, dev):
    c = W.config("toy")
    c.cfg_id = 43
    specs = _tensors()
    case = StepCase(c, tensors=[t for t, _ in specs], V=3, dev_lo=dev[0], dev_hi=dev[1])
    used = _craft(case, [r for _, r in specs], seed=100 + dev[0])
    want, seen = _modes(case)
    got = case.run_gpu(cuda)
    _compare(case, got, want)
    if dev == (0, 3):  # the whole buffer: every branch is taken somewhere
        assert used >= {NORMAL, TINY_M, TINY_V, UNDER, UNDER8}, used
        for k in ("m", "v"):
            assert seen[k] >= {"underflow", "recip", "div"}, (k, seen[k])
        assert seen["fp8"] >= {"underflow", "recip", "div"}, seen["fp8"]
    # FP8 codes of scale-0 tiles carry each element's sign
    for slot, pos in P.fp8_tiles(case.olayout, case.dev_lo, case.dev_hi):
        if want["fs"][slot] == 0:
            assert np.all((got["fp8"][pos] & 0x7F) == 0)
    _ = OF
