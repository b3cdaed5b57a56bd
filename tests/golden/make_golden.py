"""Writes the stored expected values under tests/golden/ by calling the oracle
only (plus the workload shapes).  Re-run after a justified change to the oracle:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402
from oracle import adam8 as A  # noqa: E402
from oracle import fp8 as F  # noqa: E402
from oracle import planner as P  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def layouts():
    out = {}
    for name in W.NAMED[:4] + W.SMALL[1:4]:
        c = W.config(name)
        for u in c.units:
            d = [P.TensorDesc(t.rows, t.cols, t.g, t.adam_kind, t.fp8) for t in u.tensors]
            L = P.plan(d, c.V, c.alpha, c.start_align)
            ex = L.export()
            out[f"{name}/{u.name}"] = dict(V=c.V, S=L.S, NI=len(L.intervals), n_mslots=L.n_mslots,
                                           n_fslots=L.n_fslots, starts=L.starts,
                                           export_sum=int(np.sum(np.asarray(ex, np.int64) % 1000003)))
    return out


def tiny_blocks():
    """A worked example small enough to read: one 256-element Adam block and one
    FP8 tile of its updated parameters, from fixed seeded inputs."""
    rng = np.random.default_rng(2024)
    g = (rng.standard_normal(256) * 1e-3).astype(np.float32)
    gb = torch.from_numpy(g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    p = (rng.standard_normal(256) * 0.02).astype(np.float32)
    qm = rng.integers(-127, 128, 256).astype(np.int8)
    qv = rng.integers(64, 256, 256).astype(np.uint8)
    hp = A.adam_hparams(1e-3, 0.9, 0.999, 1e-8, 10)
    p1, qm1, qv1, sm1, sv1 = A.adam8_block(gb, p, qm, qv, np.float32(1e-5), np.float32(4e-9), hp)
    q8, s8 = F.fp8_tile(p1[:128])
    return dict(grad_bits=gb.tolist(), p=p.view(np.uint32).tolist(), qm=qm.tolist(), qv=qv.tolist(),
                sm=float(np.float32(1e-5)), sv=float(np.float32(4e-9)),
                out_p=p1.view(np.uint32).tolist(), out_qm=qm1.tolist(), out_qv=qv1.tolist(),
                out_sm=int(np.float32(sm1).view(np.uint32)), out_sv=int(np.float32(sv1).view(np.uint32)),
                fp8_codes=q8.tolist(), fp8_scale=int(np.float32(s8).view(np.uint32)))


if __name__ == "__main__":
    with open(os.path.join(HERE, "layouts.json"), "w") as f:
        json.dump(layouts(), f, indent=1, sort_keys=True)
    with open(os.path.join(HERE, "adam8_fp8_block.json"), "w") as f:
        json.dump(tiny_blocks(), f)
    print("wrote", os.listdir(HERE))
