"""The DBuffer step of several units captured in one CUDA graph: replaying the
graph gives bit for bit what the same calls give launched one by one (and the
eager result is the oracle's, checked elsewhere).  Covers the TMA-fed strip
kernel, the 128x128 and 32x32 tile kernels and the flat kernels inside a graph."""

import numpy as np
import pytest
import torch

import block_quant_gb300 as bq
import workloads as W
from _step_harness import StepCase, assert_bits_equal

pytestmark = pytest.mark.gpu


class DeviceUnit:
    """Device copies of one StepCase's inputs (each call mutates them in place)."""

    def __init__(self, case, dev):
        d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        self.ws = torch.empty(case.layout.upload_bytes(case.dev_lo, case.dev_hi), dtype=torch.uint8, device=dev)
        self.shard = case.layout.upload(case.dev_lo, case.dev_hi, self.ws)
        self.gbufs, ptrs = [], np.zeros(len(case.unit.tensors), np.int64)
        for i, (bits, lo) in case.grads.items():
            g = d(bits.view(np.int16))
            self.gbufs.append(g)
            ptrs[i] = g.data_ptr() - 2 * lo
        self.gp = d(ptrs)
        self.dbuf = d(case.dbuf0.view(np.int16))
        self.master, self.m, self.v = d(case.master), d(case.m), d(case.v)
        self.ms, self.vs = d(case.ms), d(case.vs)
        self.fp8, self.fs = d(case.fp8_0), d(case.fs0)
        self.scale, self.hp = 1.0 / case.V, case.hp_c

    def step(self, stream):
        bq.pack(self.shard, self.gp, self.dbuf, self.scale, False, stream=stream)
        bq.step_adam8(self.shard, self.dbuf, self.master, self.m, self.v, self.ms, self.vs, self.hp,
                      self.fp8, self.fs, stream=stream)

    def outputs(self):
        return {k: getattr(self, k).cpu().numpy() for k in ("dbuf", "master", "m", "v", "ms", "vs", "fp8", "fs")}


def test_model_step_graph_replay_matches_eager(cuda):
    cases = [StepCase(W.config(n)) for n in ("llama-small", "llama-tile-small", "gptoss-small", "llama-tile32-small")]
    stream = torch.cuda.Stream(cuda)
    eager = [DeviceUnit(c, cuda) for c in cases]
    graphed = [DeviceUnit(c, cuda) for c in cases]
    torch.cuda.synchronize(cuda)
    with torch.cuda.stream(stream):
        for u in eager:  # first calls also set the kernels' launch attributes
            u.step(stream)
    torch.cuda.synchronize(cuda)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for u in graphed:
            u.step(stream)
    g.replay()
    torch.cuda.synchronize(cuda)
    for c, a, b in zip(cases, eager, graphed):
        bq.shard_check(a.shard)
        bq.shard_check(b.shard)
        oa, ob = a.outputs(), b.outputs()
        for k in oa:
            assert_bits_equal(f"{c.cfg.name} {k}", ob[k], oa[k])
    # a second replay continues from the updated state exactly like a second eager step
    with torch.cuda.stream(stream):
        for u in eager:
            u.step(stream)
    g.replay()
    torch.cuda.synchronize(cuda)
    for c, a, b in zip(cases, eager, graphed):
        oa, ob = a.outputs(), b.outputs()
        for k in ("master", "m", "v", "ms", "vs", "fp8", "fs"):
            assert_bits_equal(f"{c.cfg.name} {k} (step 2)", ob[k], oa[k])


def test_branched_graph_matches_eager(cuda):
    """The units captured on separate branches (side streams forked from and
    joined back to the capture stream) run concurrently in the graph and give
    bit for bit the eager results: the units share no data."""
    cases = [StepCase(W.config(n)) for n in ("llama-small", "llama-tile-small", "gptoss-small", "llama-tile32-small")]
    stream = torch.cuda.Stream(cuda)
    branches = [torch.cuda.Stream(cuda) for _ in range(3)]
    eager = [DeviceUnit(c, cuda) for c in cases]
    graphed = [DeviceUnit(c, cuda) for c in cases]
    torch.cuda.synchronize(cuda)
    with torch.cuda.stream(stream):
        for u in eager:
            u.step(stream)
    torch.cuda.synchronize(cuda)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fork = torch.cuda.Event()
        fork.record(stream)
        for b in branches:
            b.wait_event(fork)
        for i, u in enumerate(graphed):
            u.step(branches[i % len(branches)])
        for b in branches:
            join = torch.cuda.Event()
            join.record(b)
            stream.wait_event(join)
    g.replay()
    torch.cuda.synchronize(cuda)
    for c, a, b in zip(cases, eager, graphed):
        bq.shard_check(b.shard)
        oa, ob = a.outputs(), b.outputs()
        for k in oa:
            assert_bits_equal(f"{c.cfg.name} {k} (branched)", ob[k], oa[k])
