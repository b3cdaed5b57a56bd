"""The allocation-free Newton-Schulz entry point (bq_muon_ns_noalloc), for
callers that cannot allocate device memory when the step runs, against the
workspace entry point (bq_muon_ns) on the same inputs, two calls in a row.

This file sorts last so that a run stopping at the first failure has run every
other test before it."""

import numpy as np
import pytest
import torch

import block_quant_gb300 as bq
import workloads as W

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the Newton-Schulz tolerance of the parity tests


def _batch(dev, shapes, seed):
    bits = [W.muon_input_bits(seed, i, r, c) for i, (r, c) in enumerate(shapes)]
    xs = [torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16) for b in bits]
    return xs


def test_noalloc_matches_workspace_entry_point(cuda):
    shapes = [(256, 640), (384, 384), (640, 200)]  # wide, square, tall: all fit the static scratch
    for call, seed in enumerate((31, 32)):  # two calls in a row, different inputs
        xs = _batch(cuda, shapes, seed)
        y_ws = [torch.full_like(x, float("nan")) for x in xs]
        y_na = [torch.full_like(x, float("nan")) for x in xs]
        mats_ws = [(x, y, r, c) for x, y, (r, c) in zip(xs, y_ws, shapes)]
        mats_na = [(x, y, r, c) for x, y, (r, c) in zip(xs, y_na, shapes)]
        ws = torch.empty(bq.muon_ns_workspace(mats_ws), dtype=torch.uint8, device=cuda)
        bq.muon_ns(mats_ws, ws)
        bq.muon_ns_check(ws)
        bq.muon_ns_noalloc(mats_na)
        torch.cuda.synchronize(cuda)
        for (r, c), a, b in zip(shapes, y_ws, y_na):
            a64 = a.double()
            b64 = b.double()
            assert torch.isfinite(b64).all(), (call, r, c)
            rel = float(torch.linalg.norm(b64 - a64) / torch.linalg.norm(a64))
            assert rel <= TOL, (call, r, c, rel)


def test_noalloc_rejects_batches_above_the_scratch(cuda):
    x = torch.zeros(2048, 2048, dtype=torch.bfloat16, device=cuda)
    y = torch.empty_like(x)
    with pytest.raises(bq.BQError) as e:
        bq.muon_ns_noalloc([(x, y, 2048, 2048)])
    assert e.value.code == bq.BQ_ENOSPC
