"""Shared set-up for the Newton-Schulz parity tests: seeded bf16 inputs, the CUDA
path through the C ABI, the fp64 oracle on the same inputs."""

import numpy as np
import torch

import block_quant_gb300 as bq
import workloads as W
from oracle import muon as OM


def run_muon_case(dev, shapes, seed_cfg=15, steps=5, return_outputs=False):
    """Relative Frobenius error of the GPU result against the fp64 oracle, per
    matrix (all matrices go through one batched call)."""
    xs_bits = [W.muon_input_bits(seed_cfg, i, r, c) for i, (r, c) in enumerate(shapes)]
    xs = [torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16) for b in xs_bits]
    ys = [torch.full_like(x, float("nan")) for x in xs]
    mats = [(x, y, r, c) for x, y, (r, c) in zip(xs, ys, shapes)]
    ws = torch.empty(bq.muon_ns_workspace(mats), dtype=torch.uint8, device=dev)
    bq.muon_ns(mats, ws, steps=steps)
    bq.muon_ns_check(ws)
    errs, outs = [], []
    for b, y in zip(xs_bits, ys):
        x64 = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ref = OM.newton_schulz(x64, steps=steps)
        got = y.float().cpu().numpy().astype(np.float64)
        errs.append(float(np.linalg.norm(got - ref) / np.linalg.norm(ref)))
        outs.append((got, ref))
    return (errs, outs) if return_outputs else errs
