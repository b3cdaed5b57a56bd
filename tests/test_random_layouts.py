"""Seeded random units stepped as one group, every member against the oracle bit
for bit.

Each unit mixes every tensor kind the planner handles: 1-D tensors with flat
256-element blocks (with and without 1x128 FP8 tiles), 128- and 32-element tiles;
2-D tensors with flat blocks and no FP8, 128-row bands whose blocks cross rows
(C % 256 != 0) and 256-column strips (C % 256 == 0) with 128x128 FP8 tiles,
128x128 and 32x32 Adam tiles, and Muon matrices (left alone by the Adam step).
Shapes, the number of virtual devices and each member's device range are drawn
from a seeded generator, so tensors are cut at irregular offsets by the device
boundaries, bands and tiles are ragged and last blocks are short: the irregular
per-device intervals that the GPT-OSS-120B configuration's secondary run calls
for, on every kernel family at once."""

import copy

import numpy as np
import pytest

import workloads as W
from _step_harness import StepCase, assert_bits_equal, run_group_gpu

pytestmark = pytest.mark.gpu

T = W.TensorSpec


def _tensor(rng, i):
    """One random tensor of a random kind (sizes kept small for the oracle)."""
    kind = int(rng.integers(0, 9))
    yes = bool(rng.integers(0, 2))
    if kind == 0:  # 1-D, flat 256-element blocks, FP8 1x128 tiles or none
        return T(f"f{i}", 1, int(rng.integers(1, 5000)), 256, W.ADAM_FLAT256, yes)
    if kind == 1:  # 1-D, 128-element tiles
        return T(f"t{i}", 1, int(rng.integers(1, 3000)), 128, W.ADAM_TILE128, yes)
    if kind == 2:  # 1-D, 32-element tiles
        return T(f"s{i}", 1, int(rng.integers(1, 2000)), 32, W.ADAM_TILE32, False)
    rows = int(rng.integers(2, 300))
    if kind == 3:  # 2-D, flat blocks, no FP8
        cols = 8 * int(rng.integers(1, 90))
        return T(f"p{i}", rows, cols, 256 * int(rng.integers(1, 4)), W.ADAM_FLAT256, False)
    if kind == 4:  # 2-D band: blocks cross rows
        c8 = int(rng.integers(1, 90))
        cols = 8 * (c8 if c8 % 32 else c8 + 1)
        return T(f"b{i}", rows, cols, 128 * cols, W.ADAM_FLAT256, True)
    if kind == 5:  # 2-D 256-column strips
        cols = 256 * int(rng.integers(1, 4))
        return T(f"r{i}", rows, cols, 128 * cols, W.ADAM_FLAT256, True)
    if kind == 6:  # 2-D 128x128 Adam tiles, with or without FP8
        cols = 8 * int(rng.integers(1, 60))
        return T(f"q{i}", rows, cols, 128 * cols, W.ADAM_TILE128, yes)
    if kind == 7:  # 2-D 32x32 Adam tiles
        cols = 8 * int(rng.integers(1, 60))
        return T(f"w{i}", rows, cols, 32 * cols, W.ADAM_TILE32, False)
    cols = 8 * int(rng.integers(1, 40))  # Muon matrix, whole-row granularity
    return T(f"u{i}", rows, cols, rows * cols, W.OPT_MUON, False)


def _cases(seed):
    rng = np.random.default_rng([seed, 4242])
    cases = []
    for u in range(3):
        cfg = copy.deepcopy(W.config("toy"))
        cfg.cfg_id = 300 + 10 * seed + u
        tensors = [_tensor(rng, i) for i in range(int(rng.integers(4, 10)))]
        V = int(rng.integers(1, 8))
        lo = int(rng.integers(0, V))
        hi = int(rng.integers(lo + 1, V + 1))
        cases.append(StepCase(cfg, tensors=tensors, V=V, dev_lo=lo, dev_hi=hi))
    return cases


@pytest.mark.parametrize("seed", [0, 1, 2, 3, 6, 7, 8, 9])
def test_random_units_as_one_group(cuda, seed):
    cases = _cases(seed)
    scale = 0.25
    outs, gaps, _ = run_group_gpu(cases, cuda, scale)
    for c, got in zip(cases, outs):
        want = c.run_oracle(scale=scale)
        for k in ("dbuf", "master", "m", "v", "ms", "vs", "fp8"):
            assert_bits_equal(f"seed {seed} {c.cfg.cfg_id} {k}", got[k], want[k])
        assert_bits_equal(f"seed {seed} {c.cfg.cfg_id} fp8 scales", got["fs"], want["fs"][:c.nf])
        assert_bits_equal(f"seed {seed} {c.cfg.cfg_id} fp8 (standalone)", got["q2"], want["fp8"])
    assert not gaps["dbuf"].any()


@pytest.mark.parametrize("seed", [4, 5])
def test_random_units_without_fp8_output(cuda, seed):
    """fp8_out = NULL over the same kind of random group: every kernel family's
    no-FP8 instantiation, Adam state and master bit for bit."""
    cases = _cases(seed)
    outs, _, _ = run_group_gpu(cases, cuda, 1.0, fp8=False)
    for c, got in zip(cases, outs):
        want = c.run_oracle(scale=1.0)
        for k in ("dbuf", "master", "m", "v", "ms", "vs"):
            assert_bits_equal(f"seed {seed} {c.cfg.cfg_id} {k}", got[k], want[k])
