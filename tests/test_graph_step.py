"""The DBuffer step of several units captured in one CUDA graph: replaying the
graph gives bit for bit the oracle's result (and what the same calls give
launched one by one); a second replay equals the oracle's second step.  Covers
the TMA-fed strip kernel, the 128x128 and 32x32 tile kernels and the flat
kernels inside a graph, serial and on branches.  A captured step's strip kernel
copies block by block, while the eager units' steps read through the tensor
maps built for their buffers: the two stagings are held to each other and to
the oracle bit for bit."""

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
        out = {k: getattr(self, k).cpu().numpy() for k in ("dbuf", "master", "m", "v", "ms", "vs", "fp8", "fs")}
        out["dbuf"] = out["dbuf"].view(np.uint16)
        return out


def _oracle_two_steps(case):
    """The oracle's first step, and its second step from the first one's state
    (same gradients, same hyper-parameters, as a replay does)."""
    from oracle import adam8 as OA
    from oracle import fp8 as OF

    one = case.run_oracle()
    L, lo, hi = case.olayout, case.dev_lo, case.dev_hi
    master, m, v, ms, vs = OA.adam8_step(L, lo, hi, one["dbuf"], one["master"], one["m"], one["v"], one["ms"],
                                         one["vs"], case.hp_o)
    q, fs = OF.quant_fp8(L, lo, hi, master, one["fp8"], one["fs"])
    two = dict(dbuf=one["dbuf"], master=master, m=m, v=v, ms=ms, vs=vs, fp8=q, fs=fs)
    return one, two


def _check_against(name, got, want):
    for k in ("dbuf", "master", "m", "v", "ms", "vs", "fp8", "fs"):
        assert_bits_equal(f"{name} {k}", got[k], want[k])


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
    oracle = [_oracle_two_steps(c) for c in cases]
    for c, a, b, (one, _) in zip(cases, eager, graphed, oracle):
        bq.shard_check(a.shard)
        bq.shard_check(b.shard)
        oa, ob = a.outputs(), b.outputs()
        _check_against(f"{c.cfg.name} graph vs oracle", ob, one)
        for k in oa:
            assert_bits_equal(f"{c.cfg.name} {k}", ob[k], oa[k])
    # a second replay continues from the updated state: the oracle's second step
    with torch.cuda.stream(stream):
        for u in eager:
            u.step(stream)
    g.replay()
    torch.cuda.synchronize(cuda)
    for c, a, b, (_, two) in zip(cases, eager, graphed, oracle):
        oa, ob = a.outputs(), b.outputs()
        _check_against(f"{c.cfg.name} graph step 2 vs oracle", ob, two)
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
        _check_against(f"{c.cfg.name} branched graph vs oracle", ob, c.run_oracle())
        for k in oa:
            assert_bits_equal(f"{c.cfg.name} {k} (branched)", ob[k], oa[k])
