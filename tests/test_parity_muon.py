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
    # B X on CTA pairs (256-row tiles, 128 rows a CTA): the last pair tile ragged in
    # one CTA or wholly past the matrix in the other, N ragged too
    [(700, 900), (1100, 640), (300, 2000)],
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


def test_concurrent_sequential_and_graphed_batches_agree(cuda):
    """A batch with the full workspace runs its matrices concurrently on the
    library's side streams; with only the largest matrix's need it runs them one
    after another; captured in a CUDA graph the fork and join become graph
    edges.  The kernels are the same, so all three give the same bits, and each
    is within the tolerance of the fp64 oracle."""
    import torch

    import block_quant_gb300 as bq
    from oracle import muon as OM

    shapes = [(256, 640), (384, 384), (640, 200), (128, 1000)]
    bits = [W.muon_input_bits(61, i, r, c) for i, (r, c) in enumerate(shapes)]
    xs = [torch.from_numpy(b.view(np.int16)).to(cuda).view(torch.bfloat16) for b in bits]

    def batch():
        ys = [torch.full_like(x, float("nan")) for x in xs]
        return ys, [(x, y, r, c) for x, y, (r, c) in zip(xs, ys, shapes)]

    y_conc, mats = batch()
    full = bq.muon_ns_workspace(mats)
    single = max(bq.muon_ns_workspace([m]) for m in mats)
    assert full > single
    ws = torch.empty(full, dtype=torch.uint8, device=cuda)
    bq.muon_ns(mats, ws)
    bq.muon_ns_check(ws)
    y_seq, mats_s = batch()
    bq.muon_ns(mats_s, ws, ws_bytes=single)
    bq.muon_ns_check(ws)
    y_graph, mats_g = batch()
    side = torch.cuda.Stream(cuda)
    torch.cuda.synchronize(cuda)
    with torch.cuda.stream(side):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            bq.muon_ns(mats_g, ws, stream=side)
        g.replay()
    torch.cuda.synchronize(cuda)
    bq.muon_ns_check(ws)
    for (r, c), b, a, s_, gr in zip(shapes, bits, y_conc, y_seq, y_graph):
        ai = a.view(torch.int16).cpu().numpy()
        assert np.array_equal(ai, s_.view(torch.int16).cpu().numpy()), (r, c, "sequential")
        assert np.array_equal(ai, gr.view(torch.int16).cpu().numpy()), (r, c, "graph")
        x64 = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ref = OM.newton_schulz(x64, steps=5)
        got = a.float().cpu().numpy().astype(np.float64)
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < TOL, (r, c)
