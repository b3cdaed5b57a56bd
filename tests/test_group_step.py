"""Several shard ranges stepped as one group (bq_group_upload): one pack, one
Adam (+ FP8) and one standalone FP8 call over every member at once give, member
by member, the oracle's result for that member alone, bit for bit; the gaps
between members are padding (zeroed in the gradient DBuffer, untouched
elsewhere).  Covers every Adam kernel family, identical members sharing one
layout, eager launches and a CUDA graph replay."""

import copy

import numpy as np
import pytest

import workloads as W
from _step_harness import GAP_F32, GAP_I8, GAP_U8, StepCase, assert_bits_equal, run_group_gpu

pytestmark = pytest.mark.gpu


def _members():
    cases = [StepCase(W.config("llama-small")),
             StepCase(W.config("llama-tile-small"), dev_lo=1, dev_hi=3),
             StepCase(W.config("gptoss-small"), dev_lo=2, dev_hi=7),
             StepCase(W.config("toy"), dev_lo=1, dev_hi=3),
             StepCase(W.config("llama-tile32-small"), dev_lo=0, dev_hi=3),
             StepCase(W.config("muon-step-small"), dev_lo=2, dev_hi=5)]
    # an identical unit with other inputs (a second layer of the same shape)
    c2 = copy.deepcopy(W.config("llama-small"))
    c2.cfg_id = 112
    cases.append(StepCase(c2, dev_lo=3, dev_hi=6))
    return cases


SCALE = 0.125  # one pack scale for the whole group


def _compare(c, got, want, fp8=True):
    for k in ("dbuf", "master", "m", "v", "ms", "vs"):
        assert_bits_equal(f"{c.cfg.name} {k}", got[k], want[k])
    if fp8:
        assert_bits_equal(f"{c.cfg.name} fp8", got["fp8"], want["fp8"])
        assert_bits_equal(f"{c.cfg.name} fp8 scales", got["fs"], want["fs"][:c.nf])
    assert_bits_equal(f"{c.cfg.name} fp8 (standalone)", got["q2"], want["fp8"])
    assert_bits_equal(f"{c.cfg.name} fp8 scales (standalone)", got["s2"], want["fs"][:c.nf])


@pytest.mark.parametrize("graph", [False, True])
def test_group_step_matches_oracle_per_member(cuda, graph):
    cases = _members()
    outs, gaps, grp = run_group_gpu(cases, cuda, SCALE, graph=graph)
    assert grp.info["tensors"] == sum(len(c.unit.tensors) for c in cases)
    for c, got in zip(cases, outs):
        _compare(c, got, c.run_oracle(scale=SCALE))
    assert not gaps["dbuf"].any()  # gaps are padding: zeroed by the pack
    assert np.all(gaps["master"] == GAP_F32) and np.all(gaps["m"] == GAP_I8) and np.all(gaps["v"] == GAP_U8)
    assert np.all(gaps["fp8"] == 0xAA) and np.all(gaps["q2"] == 0xAA)


def test_group_step_without_fp8_output(cuda):
    cases = _members()[:3]
    outs, _, _ = run_group_gpu(cases, cuda, SCALE, fp8=False)
    for c, got in zip(cases, outs):
        _compare(c, got, c.run_oracle(scale=SCALE), fp8=False)
