"""The allocation-free Newton-Schulz entry point (bq_muon_ns_noalloc).

Some callers cannot call cudaMalloc when the optimizer step runs: runtimes that
reserve all GPU memory up front and forbid later allocations, plug-ins whose host
framework owns the allocator, and paths that must not allocate for latency
reasons.  bq_muon_ns_noalloc serves them from a fixed scratch array inside the
library.  Here it is checked against the workspace entry point (bq_muon_ns) on
the same inputs, two calls in a row: both run the same deterministic kernels, so
the outputs must agree bit for bit; each output is also held to the fp64
oracle's tolerance, and the call's device error word (in the static scratch) is
read back clear.

This file sorts last so that a run stopping at the first failure has run every
other test before it."""

import numpy as np
import pytest
import torch

import block_quant_gb300 as bq
import workloads as W
from oracle import muon as OM

pytestmark = pytest.mark.gpu

TOL = 2e-2  # relative Frobenius error against the fp64 oracle, as in the other Newton-Schulz tests


def _batch(dev, shapes, seed):
    bits = [W.muon_input_bits(seed, i, r, c) for i, (r, c) in enumerate(shapes)]
    xs = [torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16) for b in bits]
    return bits, xs


def test_noalloc_matches_workspace_entry_point(cuda):
    shapes = [(256, 640), (384, 384), (640, 200)]  # wide, square, tall: all fit the static scratch
    for call, seed in enumerate((31, 32)):  # two calls in a row, different inputs
        bits, xs = _batch(cuda, shapes, seed)
        y_ws = [torch.full_like(x, float("nan")) for x in xs]
        y_na = [torch.full_like(x, float("nan")) for x in xs]
        mats_ws = [(x, y, r, c) for x, y, (r, c) in zip(xs, y_ws, shapes)]
        mats_na = [(x, y, r, c) for x, y, (r, c) in zip(xs, y_na, shapes)]
        ws = torch.empty(bq.muon_ns_workspace(mats_ws), dtype=torch.uint8, device=cuda)
        bq.muon_ns(mats_ws, ws)
        bq.muon_ns_check(ws)
        bq.muon_ns_noalloc(mats_na)
        bq.muon_ns_check(None)  # the static scratch's error word: no wait gave up
        torch.cuda.synchronize(cuda)
        for (r, c), b, a, y in zip(shapes, bits, y_ws, y_na):
            got = y.view(torch.int16).cpu().numpy()
            want = a.view(torch.int16).cpu().numpy()
            diff = int(np.count_nonzero(got != want))
            assert diff == 0, f"call {call}, {r}x{c}: {diff} of {got.size} outputs differ from bq_muon_ns"
            x64 = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            ref = OM.newton_schulz(x64, steps=5)
            y64 = y.float().cpu().numpy().astype(np.float64)
            rel = float(np.linalg.norm(y64 - ref) / np.linalg.norm(ref))
            assert rel <= TOL, (call, r, c, rel)


def test_noalloc_rejects_batches_above_the_scratch(cuda):
    x = torch.zeros(2048, 2048, dtype=torch.bfloat16, device=cuda)
    y = torch.empty_like(x)
    with pytest.raises(bq.BQError) as e:
        bq.muon_ns_noalloc([(x, y, 2048, 2048)])
    assert e.value.code == bq.BQ_ENOSPC
