#!/usr/bin/env python
"""Benchmark of the GB300 DBuffer step (one JSON line on rank 0).

One step = the hot path over one batch of synthetic input:
  * the DBuffer step of one Llama-3-8B-shaped decoder layer held in one DBuffer
    of V = 8 simulated devices (all 8 local shards, 218.1 M parameters):
    bq_pack (fused pre-communication copy/scale/zero into the bf16 gradient
    buffer) then bq_step_adam8 (block-wise 8-bit Adam fused with 128x128 FP8
    requantisation into the AllGather staging buffer);
  * Muon's Newton-Schulz (5 iterations) on the batch of whole matrices
    4096x4096, 4096x14336, 14336x4096 (when --muon is on).
value = algorithmic DBuffer bytes per step / DBuffer time per step (GB/s);
the Muon part is reported beside it in TFLOP/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): one rank per GPU, each processes its own layer (weak
scaling, no collective on the data path); value sums the ranks' bytes over the
slowest rank's time.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "DBuffer step GB/s & fraction of HBM peak; Muon NS TFLOP/s (1 GB300)"
WORKLOAD = "llama3-8b-layer"
MUON = "muon-ns"
L2_BYTES = 126 * 2 ** 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def recorded_traffic(call):
    """DRAM bytes per launch of `call` from the committed ncu record, or None when
    the kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(call)
    if not rec:
        return None
    paths = [os.path.join(ROOT, name) for name in rec["sources"]]
    if not all(os.path.exists(q) for q in paths):
        return None
    return rec["traffic_bytes_per_launch"] if code_digest(paths) == rec["code_sha256"] else None


def code_digest(paths):
    """sha256 over C/C++/CUDA sources with comments and blank lines removed, so
    that the record follows the code, not its commentary."""
    import hashlib
    import re

    h = hashlib.sha256()
    for q in paths:
        text = re.sub(r"/\*.*?\*/", "", open(q).read(), flags=re.S)
        for line in text.splitlines():
            # a // comment: the first // that is not inside a string literal
            out, quoted = [], False
            for i, ch in enumerate(line):
                if ch == '"' and (i == 0 or line[i - 1] != "\\"):
                    quoted = not quoted
                if not quoted and line.startswith("//", i):
                    break
                out.append(ch)
            code = "".join(out).rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()


# ----------------------------------------------------------------------------- algorithmic bytes

def step_bytes(table, dev_lo, dev_hi):
    """Algorithmic DRAM bytes of one DBuffer step over local shards [dev_lo, dev_hi).
    pack: read bf16 grad 2 + write bf16 DBuffer 2 per element, +2 per padding
    element (zeroed); adam8 + FP8: grad 2 + master 4+4 + m 1+1 + v 1+1 + fp8 1
    = 15 per element, + 16 B per Adam block (two fp32 scales read and written)
    + 4 B per FP8 tile (scale written)."""
    iv = table.dev_intervals(dev_lo, dev_hi)
    elems = int(iv[:, 3].sum())
    total = (dev_hi - dev_lo) * table.S
    pads = total - elems
    m0, m1 = table.slot_range(dev_lo, dev_hi)
    f0, f1 = table.slot_range(dev_lo, dev_hi, fp8=True)
    fp8_elems = adam_elems = 0
    for k, i, t_off, ln, loff, ms, fs in iv:
        if fs >= 0:
            fp8_elems += int(ln)
        if table.tensors[i][5] != W.OPT_MUON:  # Muon tensors are not touched by the Adam step
            adam_elems += int(ln)
    pack = 4 * elems + 2 * pads
    adam = 14 * adam_elems + fp8_elems + 16 * (m1 - m0) + 4 * (f1 - f0)
    return dict(elems=elems, pads=pads, pack=pack, adam=adam, total=pack + adam,
                adam_blocks=m1 - m0, fp8_tiles=f1 - f0)


def adam_launches(table, dev_lo, dev_hi):
    """Kernels one bq_step_adam8 call launches (one per non-empty group kind)."""
    kinds = set()
    for k, i, t_off, ln, loff, ms, fs in table.dev_intervals(dev_lo, dev_hi):
        _, _, rows, cols, g, kind, fp8 = table.tensors[i]
        if kind == W.OPT_MUON:
            continue
        if kind == W.ADAM_TILE32:
            kinds.add("flat32" if rows == 1 else "tile32")
        elif kind == W.ADAM_FLAT256 and (rows == 1 or not fp8):
            kinds.add("flat256")
        elif kind == W.ADAM_TILE128 and rows == 1:
            kinds.add("flat128")
        elif kind == W.ADAM_TILE128:
            kinds.add("tile")
        else:
            kinds.add("strip")
    return len(kinds)


def muon_flops(shapes, steps=5):
    """Nominal FLOPs of the iteration: per step X X^T (2 m^2 n), A A (2 m^3),
    B X (2 m^2 n), m = min dim, n = max dim."""
    tot = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        tot += steps * (4 * m * m * n + 2 * m ** 3)
    return tot


def muon_executed_flops(shapes, steps=5, bm=128, bn=256):
    """FLOPs the tensor cores execute per batch: whole 128 x 256 tiles, and for the
    two symmetric products (X X^T, A A^T) only the tiles that touch the upper
    triangle (the kernel mirrors them)."""
    tot = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        mt, nt_sym, nt_x = -(-m // bm), -(-m // bn), -(-n // bn)
        sym = sum(1 for by in range(mt) for bx in range(nt_sym) if bx * bn + bn > by * bm)
        tile = 2 * bm * bn
        tot += steps * (sym * tile * n + sym * tile * m + mt * nt_x * tile * m)
    return tot


# ----------------------------------------------------------------------------- ranks


def max_over_ranks(vals, world, device=None):
    """Element-wise maximum of per-rank timings over all ranks (the slowest rank
    sets the job's time)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank, world, ms):
    """Whole-job rate: every rank processed units_per_rank units (weak scaling)
    in at most ms milliseconds."""
    return world * units_per_rank / (ms * 1e-3)


# ----------------------------------------------------------------------------- clocks

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            self.path = os.path.join("/tmp", f"bq_clocks_{os.getpid()}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- our arm

class DBufferStep:
    """Device-resident buffers of one unit's DBuffer step (all V local shards)."""

    def __init__(self, cfg, dev, seed, shards=None):
        import torch

        import block_quant_gb300 as bq

        self.bq, self.torch, self.dev = bq, torch, dev
        unit = cfg.units[0]
        self.V, self.lo, self.hi = cfg.V, cfg.dev_lo, cfg.dev_hi
        if shards:
            self.hi = self.lo + shards
        self.layout = bq.plan(unit.tensors, cfg.V, cfg.alpha, cfg.start_align)
        self.table = W.Table(self.layout.export())
        S = self.table.S
        n = (self.hi - self.lo) * S
        self.n = n
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        m0, m1 = self.table.slot_range(self.lo, self.hi)
        f0, f1 = self.table.slot_range(self.lo, self.hi, fp8=True)
        self.ws = torch.empty(self.layout.upload_bytes(self.lo, self.hi), dtype=torch.uint8, device=dev)
        self.shard = self.layout.upload(self.lo, self.hi, self.ws)
        # synthetic inputs with the recipe's distributions, drawn on the device
        self.master = torch.randn(n, generator=g, device=dev) * 0.02
        self.m = torch.randint(-127, 128, (n,), generator=g, device=dev, dtype=torch.int8)
        self.v = torch.randint(64, 256, (n,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        self.ms = (torch.rand(m1 - m0, generator=g, device=dev) + 0.5) * (1e-3 / 127)
        self.vs = (torch.rand(m1 - m0, generator=g, device=dev) + 0.5) * (1e-6 / 255)
        self.dbuf = torch.empty(n, dtype=torch.bfloat16, device=dev)
        self.fp8 = torch.zeros(n, dtype=torch.uint8, device=dev)
        self.fs = torch.zeros(max(f1 - f0, 1), dtype=torch.float32, device=dev)
        # per-tensor gradients over the owned ranges (distinct allocations)
        self.grads, self.host_grads, ptrs = {}, {}, np.zeros(len(unit.tensors), np.int64)
        for i in range(len(unit.tensors)):
            a, b = self.table.owned_range(i, self.lo, self.hi)
            if b > a:
                gr = (torch.randn(b - a, generator=g, device=dev) * 1e-3).to(torch.bfloat16)
                self.grads[i] = gr
                ptrs[i] = gr.data_ptr() - 2 * a
        self.gptrs = torch.from_numpy(ptrs).to(dev)
        self.hp = bq.adam_hparams(cfg.lr, cfg.b1, cfg.b2, cfg.eps, cfg.t)
        self.bytes = step_bytes(self.table, self.lo, self.hi)
        self.launches = 1 + adam_launches(self.table, self.lo, self.hi)
        torch.cuda.synchronize(dev)

    def pack(self, stream):
        self.bq.pack(self.shard, self.gptrs, self.dbuf, 1.0 / self.V, False, stream=stream)

    def adam(self, stream):
        self.bq.step_adam8(self.shard, self.dbuf, self.master, self.m, self.v, self.ms, self.vs, self.hp,
                           self.fp8, self.fs, stream=stream)

    def pin_host(self):
        torch = self.torch
        self.host_grads = {i: torch.empty(g.numel(), dtype=torch.bfloat16, pin_memory=True) for i, g in self.grads.items()}
        for i, g in self.grads.items():
            self.host_grads[i].copy_(g)
        self.host_fp8 = torch.empty(self.fp8.numel(), dtype=torch.uint8, pin_memory=True)
        self.host_fs = torch.empty(self.fs.numel(), dtype=torch.float32, pin_memory=True)
        self.h2d = sum(g.numel() * 2 for g in self.grads.values())
        self.d2h = self.fp8.numel() + self.fs.numel() * 4


class E2EPipeline:
    """End-to-end DBuffer steps through the public API from host buffers: every
    step uploads its gradients from pinned host memory, packs, runs Adam + FP8
    and reads the FP8 staging buffer and scales back.  Uploads and read-backs run
    on their own streams so that step k+1's upload and step k's read-back overlap
    step k's kernels; gradients and FP8 outputs are double-buffered, and events
    keep every buffer from being reused before its reader is done."""

    def __init__(self, step, dev):
        torch = self.torch = step.torch
        self.step, self.bq = step, step.bq
        step.pin_host()
        T, lo, hi = step.table, step.lo, step.hi
        second, ptrs = {}, np.zeros(len(step.gptrs), np.int64)
        for i, g in step.grads.items():
            a, _ = T.owned_range(i, lo, hi)
            second[i] = torch.empty_like(g)
            ptrs[i] = second[i].data_ptr() - 2 * a
        self.gsets = [step.grads, second]
        self.gptrs = [step.gptrs, torch.from_numpy(ptrs).to(dev)]
        self.fp8 = [step.fp8, torch.empty_like(step.fp8)]
        self.fs = [step.fs, torch.empty_like(step.fs)]
        self.up, self.down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]  # noqa: E731
        self.ev_up, self.ev_packed, self.ev_adam, self.ev_down = ev(), ev(), ev(), ev()
        self.k = 0

    def issue(self, comp):
        st, bq, torch, j = self.step, self.bq, self.torch, self.k & 1
        self.up.wait_event(self.ev_packed[j])  # the pack two steps back has read this set
        with torch.cuda.stream(self.up):
            for i, g in self.gsets[j].items():
                g.copy_(st.host_grads[i], non_blocking=True)
            self.ev_up[j].record(self.up)
        comp.wait_event(self.ev_up[j])
        bq.pack(st.shard, self.gptrs[j], st.dbuf, 1.0 / st.V, False, stream=comp)
        self.ev_packed[j].record(comp)
        comp.wait_event(self.ev_down[j])  # the read-back two steps back is done with this output
        bq.step_adam8(st.shard, st.dbuf, st.master, st.m, st.v, st.ms, st.vs, st.hp, self.fp8[j], self.fs[j],
                      stream=comp)
        self.ev_adam[j].record(comp)
        self.down.wait_event(self.ev_adam[j])
        with torch.cuda.stream(self.down):
            st.host_fp8.copy_(self.fp8[j], non_blocking=True)
            st.host_fs.copy_(self.fs[j], non_blocking=True)
            self.ev_down[j].record(self.down)
        self.k += 1

    def measure(self, comp, steps, warmup=3):
        torch = self.torch
        for _ in range(warmup):
            self.issue(comp)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        for _ in range(steps):
            self.issue(comp)
        comp.wait_stream(self.up)
        comp.wait_stream(self.down)
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps


class MuonBatch:
    def __init__(self, shapes, dev, seed):
        import torch

        import block_quant_gb300 as bq

        self.bq, self.torch = bq, torch
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.xs = [(torch.randn(r, c, generator=g, device=dev) * 1e-3).to(torch.bfloat16) for r, c in shapes]
        self.ys = [torch.empty_like(x) for x in self.xs]
        self.mats = [(x, y, r, c) for (x, y, (r, c)) in zip(self.xs, self.ys, shapes)]
        self.ws = torch.empty(bq.muon_ns_workspace(self.mats), dtype=torch.uint8, device=dev)
        self.flops = muon_flops(shapes)
        self.shapes = list(shapes)
        self.launches = None

    def run(self, stream):
        self.bq.muon_ns(self.mats, self.ws, stream=stream)

    def pin_host(self):
        torch = self.torch
        self.hx = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x) for x in self.xs]
        self.hy = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for y in self.ys]
        self.h2d = sum(x.numel() * 2 for x in self.xs)
        self.d2h = sum(y.numel() * 2 for y in self.ys)

    def e2e(self, comp):
        """One batch end to end from host buffers, matrix by matrix: matrix i+1's
        upload and matrix i-1's read-back overlap matrix i's Newton-Schulz (own
        streams; events keep each buffer until its reader is done)."""
        torch, n = self.torch, len(self.xs)
        if not hasattr(self, "up"):
            dev = self.xs[0].device
            self.up, self.down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
            self.ev_up, self.ev_ns, self.ev_down = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
        for i in range(n):
            self.up.wait_event(self.ev_ns[i])  # the previous batch has read x_i
            with torch.cuda.stream(self.up):
                self.xs[i].copy_(self.hx[i], non_blocking=True)
                self.ev_up[i].record(self.up)
        for i in range(n):
            comp.wait_event(self.ev_up[i])
            comp.wait_event(self.ev_down[i])  # the previous batch's y_i has been read back
            self.bq.muon_ns([self.mats[i]], self.ws, stream=comp)
            self.ev_ns[i].record(comp)
            self.down.wait_event(self.ev_ns[i])
            with torch.cuda.stream(self.down):
                self.hy[i].copy_(self.ys[i], non_blocking=True)
                self.ev_down[i].record(self.down)

    def measure_e2e(self, comp, steps=5, warmup=2):
        torch = self.torch
        for _ in range(warmup):
            self.e2e(comp)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        for _ in range(steps):
            self.e2e(comp)
        comp.wait_stream(self.up)
        comp.wait_stream(self.down)
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps


class ModelStep:
    """The DBuffer step of every unit of a model's rank-0 slice (one DBuffer per
    unit: embedding, each layer, head), each unit instance with its own buffers;
    identical units share one upload of the work tables."""

    def __init__(self, name, dev, seed):
        import torch

        import block_quant_gb300 as bq

        self.bq, self.torch = bq, torch
        cfg = W.config(name)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.units, self.bytes, self.launches, self.elems = [], 0, 0, 0
        self.keep = []
        for u in cfg.units:
            layout = bq.plan(u.tensors, cfg.V, cfg.alpha, cfg.start_align)
            T = W.Table(layout.export())
            lo, hi = cfg.dev_lo, cfg.dev_hi
            ws = torch.empty(layout.upload_bytes(lo, hi), dtype=torch.uint8, device=dev)
            shard = layout.upload(lo, hi, ws)
            self.keep += [layout, ws, shard]
            b = step_bytes(T, lo, hi)
            m0, m1 = T.slot_range(lo, hi)
            f0, f1 = T.slot_range(lo, hi, fp8=True)
            n = (hi - lo) * T.S
            for _ in range(u.repeat):
                grads, ptrs = [], np.zeros(len(u.tensors), np.int64)
                for i in range(len(u.tensors)):
                    a, bb = T.owned_range(i, lo, hi)
                    if bb > a:
                        gr = (torch.randn(bb - a, generator=g, device=dev) * 1e-3).to(torch.bfloat16)
                        grads.append(gr)
                        ptrs[i] = gr.data_ptr() - 2 * a
                unit = dict(
                    shard=shard, grads=grads, gp=torch.from_numpy(ptrs).to(dev),
                    dbuf=torch.empty(n, dtype=torch.bfloat16, device=dev),
                    master=torch.randn(n, generator=g, device=dev) * 0.02,
                    m=torch.randint(-127, 128, (n,), generator=g, device=dev, dtype=torch.int8),
                    v=torch.randint(64, 256, (n,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8),
                    ms=(torch.rand(max(m1 - m0, 1), generator=g, device=dev) + 0.5) * (1e-3 / 127),
                    vs=(torch.rand(max(m1 - m0, 1), generator=g, device=dev) + 0.5) * (1e-6 / 255),
                    fp8=torch.zeros(n, dtype=torch.uint8, device=dev),
                    fs=torch.zeros(max(f1 - f0, 1), dtype=torch.float32, device=dev),
                    V=cfg.V)
                self.units.append(unit)
                self.bytes += b["total"]
                self.elems += b["elems"]
                self.launches += 1 + adam_launches(T, lo, hi)
        self.hp = bq.adam_hparams(cfg.lr, cfg.b1, cfg.b2, cfg.eps, cfg.t)
        self.name = name

    def run(self, stream):
        bq = self.bq
        for u in self.units:
            bq.pack(u["shard"], u["gp"], u["dbuf"], 1.0 / u["V"], False, stream=stream)
            bq.step_adam8(u["shard"], u["dbuf"], u["master"], u["m"], u["v"], u["ms"], u["vs"], self.hp,
                          u["fp8"], u["fs"], stream=stream)

    def run_branches(self, stream, branches):
        """The units spread round robin over side streams forked from and joined
        back to `stream` (the units are independent), so that one unit's kernel
        tail overlaps the next unit's kernels."""
        torch, bq = self.torch, self.bq
        fork = torch.cuda.Event()
        fork.record(stream)
        for b in branches:
            b.wait_event(fork)
        for i, u in enumerate(self.units):
            b = branches[i % len(branches)]
            bq.pack(u["shard"], u["gp"], u["dbuf"], 1.0 / u["V"], False, stream=b)
            bq.step_adam8(u["shard"], u["dbuf"], u["master"], u["m"], u["v"], u["ms"], u["vs"], self.hp,
                          u["fp8"], u["fs"], stream=b)
        for b in branches:
            join = torch.cuda.Event()
            join.record(b)
            stream.wait_event(join)

    def measure(self, stream, steps=10, warmup=3):
        """(eager ms, graph ms, 4-branch graph ms) per whole-model step."""
        torch = self.torch
        eager = time_call(lambda: self.run(stream), stream, steps, warmup)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self.run(stream)
        replay = time_call(graph.replay, stream, steps, warmup)
        branches = [torch.cuda.Stream(stream.device) for _ in range(4)]
        graph4 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph4, stream=stream):
            self.run_branches(stream, branches)
        replay4 = time_call(graph4.replay, stream, steps, warmup)
        for u in self.units[:1] + self.units[-1:]:
            self.bq.shard_check(u["shard"], stream=stream)
        del graph, graph4
        return eager, replay, replay4


def time_call(fn, stream, steps, warmup):
    """Mean milliseconds of fn() on stream (CUDA events)."""
    import torch

    for _ in range(warmup):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_dbuffer(step, stream, steps, warmup):
    """Mean pack and Adam milliseconds of a DBufferStep (CUDA events)."""
    import torch

    for _ in range(warmup):
        step.pack(stream)
        step.adam(stream)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    for e in evs:
        e[0].record(stream)
        step.pack(stream)
        e[1].record(stream)
        step.adam(stream)
        e[2].record(stream)
    torch.cuda.synchronize()
    step.bq.shard_check(step.shard, stream=stream)
    return (statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
            statistics.mean(e[1].elapsed_time(e[2]) for e in evs))


class MuonStep:
    """The Muon step on the Llama-3-8B layer with its seven matrices on Muon (all
    8 shards): momentum + gather, Newton-Schulz on the gathered matrices, apply."""

    def __init__(self, dev, seed):
        import torch

        import block_quant_gb300 as bq

        self.bq, self.torch = bq, torch
        cfg = W.config("llama3-8b-layer-muon")
        unit = cfg.units[0]
        self.layout = bq.plan(unit.tensors, cfg.V, cfg.alpha, cfg.start_align)
        T = W.Table(self.layout.export())
        n = cfg.V * T.S
        self.ws = torch.empty(self.layout.upload_bytes(0, cfg.V), dtype=torch.uint8, device=dev)
        self.shard = self.layout.upload(0, cfg.V, self.ws)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.dbuf = (torch.randn(n, generator=g, device=dev) * 1e-3).to(torch.bfloat16)
        self.mom = torch.randn(n, generator=g, device=dev) * 1e-3
        self.master = torch.randn(n, generator=g, device=dev) * 0.02
        muon = [i for i, t in enumerate(unit.tensors) if t.adam_kind == W.OPT_MUON]
        shapes = [(unit.tensors[i].rows, unit.tensors[i].cols) for i in muon]
        self.gath = [torch.empty(r, c, dtype=torch.bfloat16, device=dev) for r, c in shapes]
        self.outs = [torch.empty_like(x) for x in self.gath]
        gp, up = np.zeros(len(unit.tensors), np.int64), np.zeros(len(unit.tensors), np.int64)
        for k, i in enumerate(muon):
            gp[i], up[i] = self.gath[k].data_ptr(), self.outs[k].data_ptr()
        self.gp, self.up = torch.from_numpy(gp).to(dev), torch.from_numpy(up).to(dev)
        self.lr = torch.full((len(unit.tensors),), cfg.muon_lr, dtype=torch.float32, device=dev)
        self.mu = cfg.mu
        self.mats = [(x, y, r, c) for x, y, (r, c) in zip(self.gath, self.outs, shapes)]
        self.nsws = torch.empty(bq.muon_ns_workspace(self.mats), dtype=torch.uint8, device=dev)
        self.elems = sum(r * c for r, c in shapes)
        self.flops = muon_flops(shapes)
        self.shapes = list(shapes)
        self.shapes = shapes
        roots = bq.muon_roots(self.layout)
        load = [0] * cfg.V
        for i in muon:
            r, c = unit.tensors[i].rows, unit.tensors[i].cols
            load[roots[i]] += 5 * (4 * min(r, c) ** 2 * max(r, c) + 2 * min(r, c) ** 3)
        self.root_tflop = [round(x / 1e12, 3) for x in load]
        self.V = cfg.V

    def run(self, stream, ev=None):
        bq = self.bq
        if ev:
            ev[0].record(stream)
        bq.muon_momentum(self.shard, self.dbuf, self.mom, self.mu, self.gp, stream=stream)
        if ev:
            ev[1].record(stream)
        bq.muon_ns(self.mats, self.nsws, steps=5, stream=stream)
        if ev:
            ev[2].record(stream)
        bq.muon_apply(self.shard, self.master, self.up, self.lr, stream=stream)
        if ev:
            ev[3].record(stream)

    def measure(self, stream, steps, warmup):
        torch = self.torch
        for _ in range(warmup):
            self.run(stream)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        torch.cuda.synchronize()
        for k in range(steps):
            self.run(stream, evs[k])
        torch.cuda.synchronize()
        self.bq.shard_check(self.shard, stream=stream)
        self.bq.muon_ns_check(self.nsws, stream=stream)
        mom = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
        ns = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
        app = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
        return mom, ns, app


def cpu_baseline(seconds=12.0):
    """The oracle, as it stands, on a bounded sample of the same workload: whole
    128-row x 256-column strips of the Llama-3-8B layer's 2-D tensors (pack
    arithmetic, the 128 Adam blocks and the two FP8 tiles of each strip), timed
    on one host core.  Returns GB/s at the same algorithmic bytes per element."""
    from oracle import adam8 as OA
    from oracle import codecs as OC
    from oracle import fp8 as OF

    cfg = W.config(WORKLOAD)
    hp = OA.adam_hparams(cfg.lr, cfg.b1, cfg.b2, cfg.eps, cfg.t)
    rng = np.random.default_rng(0)
    elems, spent, strips = 0, 0.0, 0
    sc = np.float32(1.0 / cfg.V)
    while spent < seconds:
        g = (rng.standard_normal((128, 256)) * 1e-3).astype(np.float32)
        gb = OC.f32_to_bf16_bits(g)
        p = (rng.standard_normal((128, 256)) * 0.02).astype(np.float32)
        qm = rng.integers(-127, 128, (128, 256)).astype(np.int8)
        qv = rng.integers(64, 256, (128, 256)).astype(np.uint8)
        t0 = time.perf_counter()
        packed = OC.f32_to_bf16_bits(OC.bf16_bits_to_f32(gb) * sc)
        p1 = np.empty_like(p)
        for r in range(128):
            p1[r], _, _, _, _ = OA.adam8_block(packed[r], p[r], qm[r], qv[r], np.float32(1e-5), np.float32(4e-9), hp)
        OF.fp8_tile(p1[:, :128])
        OF.fp8_tile(p1[:, 128:])
        spent += time.perf_counter() - t0
        elems += 128 * 256
        strips += 1
    bpe = 19.0 + 16.0 / 256 + 4.0 / 16384
    return dict(value=elems * bpe / spent / 1e9, unit="GB/s", cores=1, kind="oracle",
                sample=f"{strips} strips of 128x256 elements ({elems} elements) of the llama3-8b layer: "
                       f"oracle pack + 8-bit Adam + FP8, numpy, one thread, {spent:.1f} s")


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    import block_quant_gb300 as bq

    bq.load()
    cfg = W.config(WORKLOAD)
    step = DBufferStep(cfg, dev, seed=1000 + rank, shards=args.shards)
    muon = MuonBatch(W.config(MUON).muon_shapes, dev, seed=2000 + rank) if args.muon else None
    stream = torch.cuda.current_stream(dev)

    def one_step(ev=None):
        if ev:
            ev[0].record(stream)
        step.pack(stream)
        if ev:
            ev[1].record(stream)
        step.adam(stream)
        if ev:
            ev[2].record(stream)
        if muon:
            muon.run(stream)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = Clocks(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        one_step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    pack_ms = [e[0].elapsed_time(e[1]) for e in evs]
    adam_ms = [e[1].elapsed_time(e[2]) for e in evs]
    muon_ms = [e[2].elapsed_time(e[3]) for e in evs] if muon else [0.0]
    dbuf_ms = statistics.mean(p + a for p, a in zip(pack_ms, adam_ms))

    # end to end through the public API from pinned host buffers: each step's
    # gradients uploaded, pack + Adam + FP8, the FP8 staging buffer and scales
    # read back; uploads and read-backs overlap the neighbouring steps' kernels
    pipe = E2EPipeline(step, dev)
    e2e_ms = pipe.measure(stream, steps=max(10, args.steps // 2))
    muon_e2e = None
    if muon:
        muon.pin_host()
        muon_e2e = muon.measure_e2e(stream)

    # the toy configuration: 1.57 M parameters, L2-resident and launch-bound
    toy = DBufferStep(W.config("toy"), dev, seed=6000 + rank)

    def toy_call():
        toy.pack(stream)
        toy.adam(stream)

    toy_eager = time_call(toy_call, stream, steps=200, warmup=20)
    side_t = torch.cuda.Stream(dev)
    with torch.cuda.stream(side_t):
        gtoy = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gtoy, stream=side_t):
            toy.pack(side_t)
            toy.adam(side_t)
        toy_graph = time_call(gtoy.replay, side_t, steps=200, warmup=20)
    toy_info = (toy.bytes["total"], toy.launches)
    del gtoy, toy
    toy_eager, toy_graph = max_over_ranks([toy_eager, toy_graph], world, device=dev)
    models = {}
    if args.model_step:
        for mname in ("llama3-70b-rank0", "gpt-oss-120b-rank0"):
            mst = ModelStep(mname, dev, seed=5000 + rank)
            side = torch.cuda.Stream(dev)
            with torch.cuda.stream(side):
                res = max_over_ranks(list(mst.measure(side)), world, device=dev)
            models[mname] = (res, (mst.bytes, mst.elems, mst.launches, len(mst.units)))
            del mst
            torch.cuda.empty_cache()
    acc_ms = max_over_ranks([time_call(lambda: bq.pack(step.shard, step.gptrs, step.dbuf, 1.0 / step.V, True,
                                                       stream=stream), stream, steps=20, warmup=3)],
                            world, device=dev)[0]
    dq = None
    if args.dequant:
        view = torch.empty(step.n, dtype=torch.bfloat16, device=dev)

        def dq_call():
            bq.dequant_fp8(step.shard, step.fp8, step.fs, view, stream=stream)

        dq = max_over_ranks([time_call(dq_call, stream, steps=20, warmup=3)], world, device=dev)[0]
        dq_elems = int(sum(int(r[3]) for r in step.table.dev_intervals(step.lo, step.hi) if r[6] >= 0))
        del view
    t32 = None
    if args.tile32:
        st32 = DBufferStep(W.config("llama3-8b-layer-tile32"), dev, seed=4000 + rank)
        t32 = max_over_ranks(list(time_dbuffer(st32, stream, steps=20, warmup=3)), world, device=dev)
        t32_bytes = st32.bytes
        del st32
        torch.cuda.empty_cache()
    mstep = None
    if args.muon_step:
        ms_obj = MuonStep(dev, seed=3000 + rank)
        mstep = ms_obj.measure(stream, steps=5, warmup=3)
        mstep_max = max_over_ranks(list(mstep), world, device=dev)
    ms_step, dbuf_ms_max, muon_ms_max, e2e_max, muon_e2e_max = max_over_ranks(
        [total_ms / args.steps, dbuf_ms, statistics.mean(muon_ms), e2e_ms, muon_e2e or 0.0], world, device=dev)
    if rank == 0:
        pk = peaks()
        B = step.bytes["total"]
        value = job_throughput(B, world, dbuf_ms_max) / 1e9
        adam_mean = statistics.mean(adam_ms)
        adam_gbs = step.bytes["adam"] / (adam_mean * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(step.bytes, step.table.S, step.lo, step.hi, step.n, bool(muon), world),
            "hbm_frac": round(value / world / pk["hbm"], 4),
            "dbuffer_ms": round(dbuf_ms_max, 4),
            "pack": {"ms": round(statistics.mean(pack_ms), 4),
                     "GB/s": round(step.bytes["pack"] / (statistics.mean(pack_ms) * 1e-3) / 1e9, 1)},
            "roofline": {"bound": "hbm", "kernel": "bq_step_adam8 (8-bit Adam + fused FP8)",
                         "achieved": round(adam_gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                         "frac": round(adam_gbs / pk["hbm"], 4), "traffic": recorded_traffic("bq_step_adam8"),
                         "peak_source": f"{pk['src']} hbm_gbs (STREAM-style copy)",
                         "ms": round(adam_mean, 4), "algorithmic_bytes": step.bytes["adam"]},
            "e2e": {"value": round(job_throughput(B, world, e2e_max) / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": step.h2d, "d2h_bytes_per_step": step.d2h,
                    "overlap": "upload of step k+1 and read-back of step k run on their own streams during step k",
                    "ms_per_step": round(e2e_max, 4)},
            "gpu_launches": args.steps * (step.launches + (muon_launches(muon) if muon else 0)),
            "clocks": clk,
        }
        if muon:
            tf = job_throughput(muon.flops, world, muon_ms_max) / 1e12
            ex = muon_executed_flops(muon.shapes)
            ex_tf = job_throughput(ex, world, muon_ms_max) / 1e12
            line["muon"] = {"value": round(tf, 1), "unit": "TFLOP/s", "ms": round(muon_ms_max, 3),
                            "flops": muon.flops,
                            "count": "nominal 4 m^2 n + 2 m^3 per step; X X^T and A A^T are computed on "
                                     "the upper triangle and mirrored, so this is an effective rate",
                            "executed_flops": ex, "executed_TFLOP/s": round(ex_tf, 1),
                            "frac": round(ex_tf / world / pk["bf16_sus"], 4),
                            "frac_basis": "executed FLOPs (the tiles that run) / measured sustained bf16 peak",
                            "nominal_over_peak": round(tf / world / pk["bf16_sus"], 4),
                            "peak": pk["bf16_sus"], "peak_source": f"{pk['src']} bf16_tflops_sustained",
                            "e2e": {"value": round(job_throughput(muon.flops, world, muon_e2e_max) / 1e12, 1),
                                    "unit": "TFLOP/s", "h2d_bytes_per_step": muon.h2d,
                                    "d2h_bytes_per_step": muon.d2h, "ms_per_step": round(muon_e2e_max, 3)}}
        desc = {"llama3-70b-rank0": "all {u} units (embedding, 80 layers, head) of the rank-0 slice at V=64, one "
                                    "DBuffer each, 128x128 Adam tiles + FP8",
                "gpt-oss-120b-rank0": "all {u} units (embedding, 36 MoE layers, head) of the rank-0 slice at V=256, "
                                      "one DBuffer each, 256-element Adam blocks + 128x128 FP8 (d = 2880: whole-band "
                                      "regions)"}
        for mname, ((eg, gr, gr4), (mb, me, ml, mu)) in models.items():
            line.setdefault("model_step", {})[mname] = {
                "workload": f"{mname}: " + desc[mname].format(u=mu),
                "elements": me, "bytes": mb, "launches": ml,
                "eager": {"ms": round(eg, 3), "GB/s": round(mb / (eg * 1e-3) / 1e9, 1)},
                "cuda_graph": {"ms": round(gr, 3), "GB/s": round(mb / (gr * 1e-3) / 1e9, 1),
                               "frac": round(mb / (gr * 1e-3) / 1e9 / pk["hbm"], 4)},
                "cuda_graph_4_branches": {"ms": round(gr4, 3), "GB/s": round(mb / (gr4 * 1e-3) / 1e9, 1),
                                          "frac": round(mb / (gr4 * 1e-3) / 1e9 / pk["hbm"], 4)},
                "note": "measured after the timed region; not part of value",
            }
        tb_, tl_ = toy_info
        line["toy_step"] = {
            "workload": "toy 2-layer d=256 unit (1.57 M parameters, V=4, all shards): pack + 8-bit Adam, "
                        "L2-resident and launch-bound",
            "bytes": tb_, "launches": tl_,
            "eager": {"us": round(toy_eager * 1e3, 2), "GB/s": round(tb_ / (toy_eager * 1e-3) / 1e9, 1)},
            "cuda_graph": {"us": round(toy_graph * 1e3, 2), "GB/s": round(tb_ / (toy_graph * 1e-3) / 1e9, 1)},
            "note": "measured after the timed region; not part of value",
        }
        acc_bytes = 6 * step.bytes["elems"] + 2 * step.bytes["pads"]
        line["pack_accumulate"] = {
            "workload": "llama3-8b-layer pack with accumulation into the gradient DBuffer (read grad 2 + DBuffer 2, "
                        "write 2 per element; padding zeroed), all 8 shards",
            "ms": round(acc_ms, 4), "GB/s": round(acc_bytes / (acc_ms * 1e-3) / 1e9, 1),
            "frac": round(acc_bytes / (acc_ms * 1e-3) / 1e9 / pk["hbm"], 4), "bytes": acc_bytes,
            "note": "measured after the timed region; not part of value",
        }
        if dq:
            dq_bytes = 3 * dq_elems + 4 * step.bytes["fp8_tiles"]
            gb = dq_bytes / (dq * 1e-3) / 1e9
            line["dequant_view"] = {
                "workload": "llama3-8b-layer FP8 buffer -> bf16 view (code x tile scale), all 8 shards",
                "ms": round(dq, 4), "GB/s": round(gb, 1), "frac": round(gb / pk["hbm"], 4), "bytes": dq_bytes,
                "note": "measured after the timed region; not part of value",
            }
        if t32:
            pk_ms, ad_ms = t32
            gb = t32_bytes["adam"] / (ad_ms * 1e-3) / 1e9
            line["adam_tile32"] = {
                "workload": "llama3-8b-layer with the pages' 32x32 8-bit Adam blocks, 32-row granularity, no FP8 "
                            "(V=8, all shards)",
                "adam_ms": round(ad_ms, 4), "GB/s": round(gb, 1), "frac": round(gb / pk["hbm"], 4),
                "bytes": t32_bytes["adam"], "adam_blocks": t32_bytes["adam_blocks"],
                "step_GB/s": round(t32_bytes["total"] / ((pk_ms + ad_ms) * 1e-3) / 1e9, 1),
                "note": "measured after the timed region; not part of value",
            }
        if mstep:
            mo, ns, ap = mstep_max
            tf = ms_obj.flops / (ns * 1e-3) / 1e12
            gb_m = 12 * ms_obj.elems / (mo * 1e-3) / 1e9
            gb_a = 10 * ms_obj.elems / (ap * 1e-3) / 1e9
            line["muon_step"] = {
                "workload": "llama3-8b-layer, its 7 matrices on Muon (V=8, all shards): momentum + gather, "
                            "Newton-Schulz x 5 on the gathered matrices, apply",
                "ms": round(mo + ns + ap, 3), "muon_elements": ms_obj.elems,
                "momentum": {"ms": round(mo, 4), "GB/s": round(gb_m, 1), "frac": round(gb_m / pk["hbm"], 4),
                             "bytes": 12 * ms_obj.elems},
                "ns": {"ms": round(ns, 3), "TFLOP/s": round(tf, 1), "flops": ms_obj.flops,
                       "count": "nominal (effective: symmetric products run on the upper triangle)",
                       "executed_TFLOP/s": round(muon_executed_flops(ms_obj.shapes) / (ns * 1e-3) / 1e12, 1),
                       "frac": round(muon_executed_flops(ms_obj.shapes) / (ns * 1e-3) / 1e12 / pk["bf16_sus"], 4),
                       "frac_basis": "executed FLOPs / measured sustained bf16 peak"},
                "apply": {"ms": round(ap, 4), "GB/s": round(gb_a, 1), "frac": round(gb_a / pk["hbm"], 4),
                          "bytes": 10 * ms_obj.elems},
                "root_ns_tflop_per_device": ms_obj.root_tflop,
                "note": "measured after the timed region; not part of value",
            }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def muon_launches(muon, steps=5):
    """Kernels one bq_muon_ns call launches: per matrix a sum-of-squares
    reduction, its one-block finish, a scaled (transposing) copy, three GEMMs
    per step and the copy out."""
    return len(muon.mats) * (4 + 3 * steps)


def workload_config(b, S, lo, hi, n, muon, world):
    """The config object both arms print (b: step_bytes of the benchmarked range)."""
    return {
        "workload": f"llama3-8b-layer DBuffer step (V=8, local shards {lo}..{hi - 1})" +
                    (" + Muon NS batch [4096x4096, 4096x14336, 14336x4096] x 5 iterations" if muon else ""),
        "elements": b["elems"], "padding_elements": b["pads"], "S": S,
        "bytes_per_step": b["total"], "l2": f"inputs {n * 13 / 1e9:.1f} GB > L2: no flush needed",
        "parallelism": f"dp{world}: one independent layer per GPU, no data-path collective",
    }


def reference_config(args, world):
    """Our arm's config, with the layout figures from the oracle planner (no GPU)."""
    from oracle import planner as OP

    cfg = W.config(WORKLOAD)
    descs = [OP.TensorDesc(t.rows, t.cols, t.g, t.adam_kind, t.fp8) for t in cfg.units[0].tensors]
    T = W.Table(OP.plan(descs, cfg.V, cfg.alpha, cfg.start_align).export())
    lo, hi = cfg.dev_lo, cfg.dev_lo + (args.shards or (cfg.dev_hi - cfg.dev_lo))
    return workload_config(step_bytes(T, lo, hi), T.S, lo, hi, (hi - lo) * T.S, args.muon, world)


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores, same
    metric and unit, a bounded sample of the workload per step."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    per_step = []
    for _ in range(args.warmup):
        cpu_baseline(seconds=0.5)
    for _ in range(args.steps):
        per_step.append(cpu_baseline(seconds=1.0))
    vals = [x["value"] for x in per_step]
    v = statistics.mean(vals)
    line = {
        "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": reference_config(args, world),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": per_step[0]["sample"].split(":")[0] + " per step (about 1 s of CPU work)"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--muon", dest="muon", action="store_true", default=True)
    ap.add_argument("--no-muon", dest="muon", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--model-step", dest="model_step", action="store_true", default=True)
    ap.add_argument("--no-model-step", dest="model_step", action="store_false")
    ap.add_argument("--dequant", dest="dequant", action="store_true", default=True)
    ap.add_argument("--no-dequant", dest="dequant", action="store_false")
    ap.add_argument("--tile32", dest="tile32", action="store_true", default=True)
    ap.add_argument("--no-tile32", dest="tile32", action="store_false")
    ap.add_argument("--muon-step", dest="muon_step", action="store_true", default=True)
    ap.add_argument("--no-muon-step", dest="muon_step", action="store_false")
    ap.add_argument("--shards", type=int, default=None,
                    help="process only local shards [0, K) of the DBuffer (smaller case for profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
