"""CUDA Newton-Schulz (tcgen05 GEMMs) vs the fp64 oracle: relative Frobenius
error at most 2e-2 (bf16 operands and bf16 storage of X, A, B between products,
fp32 accumulation)."""

import numpy as np
import pytest

import workloads as W
from _muon_harness import run_muon_case

pytestmark = pytest.mark.gpu

TOL = 2e-2


def test_normalise_only(cuda):
    """steps = 0: the normalisation and the transpose rule alone (bf16 rounding of
    x / ||x||)."""
    errs = run_muon_case(cuda, [(256, 384), (384, 256), (200, 328)], steps=0)
    assert max(errs) < 4e-3, errs


def test_one_step(cuda):
    errs = run_muon_case(cuda, [(128, 256), (256, 256), (640, 256)], steps=1)
    assert max(errs) < TOL, errs


@pytest.mark.parametrize("shapes", [
    [(256, 256), (256, 640), (640, 256)],   # several tiles, tall input transposed
    [(200, 328), (328, 200), (72, 1000)],   # ragged edges in every dimension
    [(512, 1536)],
])
def test_five_steps(cuda, shapes):
    errs = run_muon_case(cuda, shapes, steps=5)
    assert max(errs) < TOL, errs


def test_full_size_batch(cuda):
    """The named Muon workload: 4096x4096, 4096x14336 and 14336x4096 in one batch,
    five steps, each matrix against the fp64 oracle."""
    c = W.config("muon-ns")
    errs = run_muon_case(cuda, c.muon_shapes, seed_cfg=c.cfg_id, steps=5)
    assert max(errs) < TOL, errs


def test_degenerate_inputs(cuda):
    """An all-zero matrix stays exactly zero (x / (0 + eps) = 0); one-row and
    one-column matrices (rank one: every step maps the single singular value
    through the quintic), a tiny square one and a very flat one against the fp64
    oracle."""
    import torch

    import block_quant_gb300 as bq

    x = torch.zeros(96, 160, dtype=torch.bfloat16, device=cuda)
    y = torch.full_like(x, float("nan"))
    mats = [(x, y, 96, 160)]
    ws = torch.empty(bq.muon_ns_workspace(mats), dtype=torch.uint8, device=cuda)
    bq.muon_ns(mats, ws, steps=5)
    bq.muon_ns_check(ws)
    assert not torch.isnan(y).any() and int(torch.count_nonzero(y)) == 0
    errs = run_muon_case(cuda, [(1, 64), (64, 1), (8, 8), (3, 1000)], steps=5)
    assert max(errs) < TOL, errs
