"""How far the kernels sit from the plain definition of the step.

The kernels reproduce the oracle's contract leg bit for bit (test_parity_step).
That leg's fp32 operation order (fused multiply-adds, reciprocal bias
corrections, codes from the product with a reciprocal block scale) is a reading
chosen to match the kernels' instruction form; the pages fix no order.  Here the
same GPU outputs are compared with the oracle's plain leg (oracle.plain: every
operation separate, division by the bias corrections and by the block scale),
end to end from the same inputs, and the mismatches are reported:

  * int8 m / uint8 v codes and E4M3 codes: how many differ, and the largest
    difference in code steps (must be at most 1);
  * block and tile scales: how many differ, and the largest relative difference;
  * the fp32 master: how many differ, and the largest difference relative to the
    parameter's magnitude max(|p|, |p'|) (must be at most 1e-6).

Run with ``-s`` to see the figures."""

import numpy as np
import pytest

import workloads as W
from _step_harness import StepCase
from oracle import fp8 as OF
from oracle import pack as OP
from oracle import plain as PL

pytestmark = pytest.mark.gpu

CODE_STEPS = 1
MASTER_REL = 1e-6


def _e4m3_ordinal(c):
    c = c.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def _report(name, case, got):
    L, lo, hi = case.olayout, case.dev_lo, case.dev_hi
    sc = np.float32(1.0 / case.V)
    dbuf = OP.pack(L, lo, hi, case.grads, case.dbuf0, sc, False)
    hp = PL.adam_hparams(case.cfg.lr, case.cfg.b1, case.cfg.b2, case.cfg.eps, case.t)
    master, m, v, ms, vs = PL.adam8_step(L, lo, hi, dbuf, case.master, case.m, case.v, case.ms, case.vs, hp)
    fp8, fs = PL.quant_fp8(L, lo, hi, master, case.fp8_0, case.fs0)
    # the plain FP8 formula on the kernel's own master isolates the quantiser form
    fp8_own, _ = PL.quant_fp8(L, lo, hi, got["master"], case.fp8_0, case.fs0)
    fp8_contract, _ = OF.quant_fp8(L, lo, hi, got["master"], case.fp8_0, case.fs0)
    assert np.array_equal(fp8_contract, got["fp8"])  # sanity: the kernel is the contract leg
    st = {}
    dm = np.abs(got["m"].astype(np.int32) - m.astype(np.int32))
    dv = np.abs(got["v"].astype(np.int32) - v.astype(np.int32))
    df = np.abs(_e4m3_ordinal(got["fp8"]) - _e4m3_ordinal(fp8))
    dfo = np.abs(_e4m3_ordinal(got["fp8"]) - _e4m3_ordinal(fp8_own))
    st["elements"] = int(case.n)
    st["m_codes"] = (int(np.count_nonzero(dm)), int(dm.max(initial=0)))
    st["v_codes"] = (int(np.count_nonzero(dv)), int(dv.max(initial=0)))
    st["fp8_codes"] = (int(np.count_nonzero(df)), int(df.max(initial=0)))
    st["fp8_codes_same_master"] = (int(np.count_nonzero(dfo)), int(dfo.max(initial=0)))

    def scale_diff(a, b):
        a, b = a.astype(np.float64), b.astype(np.float64)
        d = np.abs(a - b) / np.maximum(np.abs(b), 1e-300)
        return int(np.count_nonzero(a != b)), float(d.max(initial=0.0))

    st["m_scales"] = scale_diff(got["ms"], ms)
    st["v_scales"] = scale_diff(got["vs"], vs)
    nf = case.nf
    st["fp8_scales"] = scale_diff(got["fs"][:nf], fs[:nf])
    p0 = case.master.astype(np.float64)
    pg, pp = got["master"].astype(np.float64), master.astype(np.float64)
    mag = np.maximum(np.abs(p0), np.abs(pp))
    rel = np.where(pg != pp, np.abs(pg - pp) / np.maximum(mag, 1e-300), 0.0)
    st["master"] = (int(np.count_nonzero(pg != pp)), float(rel.max(initial=0.0)))
    print(f"\nplain-leg mismatch {name}: " + ", ".join(f"{k}={v}" for k, v in st.items()))
    assert st["m_codes"][1] <= CODE_STEPS and st["v_codes"][1] <= CODE_STEPS, st
    assert st["fp8_codes"][1] <= CODE_STEPS and st["fp8_codes_same_master"][1] <= CODE_STEPS, st
    assert st["master"][1] <= MASTER_REL, st
    return st


@pytest.mark.parametrize("name", ["toy", "llama-small", "llama-tile-small", "gptoss-small", "llama-tile32-small"])
def test_kernels_against_plain_leg(cuda, name):
    case = StepCase(W.config(name))
    _report(name, case, case.run_gpu(cuda))


def test_kernels_against_plain_leg_first_step(cuda):
    case = StepCase(W.config("gptoss-small"), t=1, zero_state=True)
    _report("gptoss-small t=1 zero state", case, case.run_gpu(cuda))


def test_kernels_against_plain_leg_full_layer(cuda):
    """The benchmarked Llama-3-8B layer's first two shards (54.5 M elements)."""
    case = StepCase(W.config("llama3-8b-layer"), dev_lo=0, dev_hi=2)
    _report("llama3-8b-layer shards 0-1", case, case.run_gpu(cuda))
