#!/usr/bin/env python
"""Benchmark of the GB300 DBuffer step (one JSON line on rank 0).

One step = the hot path over one batch of synthetic input:
  * the DBuffer step of the Llama-3-70B-shaped model's slice on one device of
    V = 64 (rank r's local shard of every fully_shard unit: embedding, 80
    layers, head; 1.2 G elements) stepped as ONE group: bq_pack (fused
    pre-communication copy/scale/zero into the bf16 gradient buffers) then
    bq_step_adam8 (block-wise 8-bit Adam with 128x128 state tiles fused with
    128x128 FP8 requantisation into the AllGather staging buffer), one launch
    per kernel family;
  * Muon's Newton-Schulz (5 iterations) on the batch of whole matrices
    4096x4096, 4096x14336, 14336x4096 (when --muon is on).
value = algorithmic DBuffer bytes per step / DBuffer time per step (GB/s);
the Muon part is reported beside it in TFLOP/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): one rank per GPU; rank r steps device r's shard of every
unit (weak scaling, no collective on the data path); value sums the ranks'
bytes over the slowest rank's time.
"""

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "DBuffer step GB/s & fraction of HBM peak; Muon NS TFLOP/s (1 GB300)"
WORKLOAD = "llama3-70b-rank0"
LAYER = "llama3-8b-layer"
GPTOSS = "gpt-oss-120b-rank0"
MUON = "muon-ns"
L2_BYTES = 126 * 2 ** 20
GROUP_ALIGN = 256  # elements between group members' bases (the library's member alignment)
ROOFLINE_KERNEL = {
    WORKLOAD: "bq_step_adam8 on the group (k_tile: 128x128 Adam tiles + fused FP8; k_flat<4>: the 1-D norms)",
    LAYER: "bq_step_adam8 (k_strip: 256-element Adam blocks + fused 128x128 FP8; k_flat<8>: the norms)",
    GPTOSS: "bq_step_adam8 on the group (k_strip over strips and band pieces, k_quant_region for the band FP8 "
            "tiles, k_flat<8>)",
}


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
                adam_blocks=m1 - m0, fp8_tiles=f1 - f0, fp8_elems=fp8_elems)


def adam_kinds(table, dev_lo, dev_hi, fp8_out=True):
    """Kernel families one bq_step_adam8 call launches for local shards
    [dev_lo, dev_hi) of a table (a group launches each family once)."""
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
            if cols % 256 and fp8_out:  # bands: Adam pieces, then the band FP8 tiles
                kinds.add("band_fp8")
    return kinds


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
    triangle (the only ones the kernel computes and stores)."""
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

def _fill(t, draw, chunk=1 << 27):
    """Fill a large device tensor chunk by chunk (bounded temporaries)."""
    for a in range(0, t.numel(), chunk):
        b = min(t.numel(), a + chunk)
        t[a:b].copy_(draw(b - a))


class GroupStep:
    """Device-resident buffers of a configuration's slice stepped as one group:
    every unit (identical units repeated), local shards [dev_lo, dev_hi) of
    each, in one set of group buffers; one pack and one Adam (+ FP8) call per
    step.  members limits the group to its first members (smaller cases)."""

    def __init__(self, name, dev, seed, dev_lo=None, members=None):
        import torch

        import block_quant_gb300 as bq

        self.bq, self.torch, self.dev = bq, torch, dev
        cfg = W.config(name)
        self.name, self.cfg = name, cfg
        lo = cfg.dev_lo if dev_lo is None else dev_lo
        hi = lo + (cfg.dev_hi - cfg.dev_lo)
        self.V, self.lo, self.hi = cfg.V, lo, hi
        self.layouts = [bq.plan(u.tensors, cfg.V, cfg.alpha, cfg.start_align) for u in cfg.units]
        tables = [W.Table(lay.export()) for lay in self.layouts]
        mem = [u for u, unit in enumerate(cfg.units) for _ in range(unit.repeat)]
        if members:
            mem = mem[:members]
        self.members = mem
        self.group = bq.Group([(self.layouts[u], lo, hi) for u in mem])
        info = self.group.info
        E = self.n = info["elems"]
        self.ws = torch.empty(self.group.upload_bytes(), dtype=torch.uint8, device=dev)
        self.shard = self.group.upload(self.ws)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        # synthetic inputs with the recipe's distributions, drawn on the device
        self.master = torch.empty(E, dtype=torch.float32, device=dev)
        _fill(self.master, lambda k: torch.randn(k, generator=g, device=dev) * 0.02)
        self.m = torch.empty(E, dtype=torch.int8, device=dev)
        _fill(self.m, lambda k: torch.randint(-127, 128, (k,), generator=g, device=dev, dtype=torch.int8))
        self.v = torch.empty(E, dtype=torch.uint8, device=dev)
        _fill(self.v, lambda k: torch.randint(64, 256, (k,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8))
        nm, nf = max(info["mslots"], 1), max(info["fslots"], 1)
        self.ms = (torch.rand(nm, generator=g, device=dev) + 0.5) * (1e-3 / 127)
        self.vs = (torch.rand(nm, generator=g, device=dev) + 0.5) * (1e-6 / 255)
        self.dbuf = torch.empty(E, dtype=torch.bfloat16, device=dev)
        self.fp8 = torch.zeros(E, dtype=torch.uint8, device=dev)
        self.fs = torch.zeros(nf, dtype=torch.float32, device=dev)
        # every member's gradients over their owned ranges: distinct tensors (no
        # two share an element), carved back to back out of one allocation so
        # that a step's upload from the host is one copy
        self.grads, self.grad_lo = {}, {}
        ptrs = np.zeros(max(info["tensors"], 1), np.int64)
        self.bytes = dict(elems=0, pads=0, pack=0, adam=0, total=0, adam_blocks=0, fp8_tiles=0, fp8_elems=0)
        kinds, covered, spans, nG = set(), 0, [], 0
        for u, p in zip(mem, self.group.place):
            T = tables[u]
            for i in range(T.N):
                a, b = T.owned_range(i, lo, hi)
                if b > a:
                    spans.append((p["tensor_base"] + i, nG, a, b - a))
                    nG += -(-(b - a) // 8) * 8  # 16-byte aligned starts
            for k, v in step_bytes(T, lo, hi).items():
                self.bytes[k] += v
            kinds |= adam_kinds(T, lo, hi)
            covered += (hi - lo) * T.S
        self.gbuf = torch.empty(max(nG, 8), dtype=torch.bfloat16, device=dev)
        _fill(self.gbuf, lambda k: (torch.randn(k, generator=g, device=dev) * 1e-3).to(torch.bfloat16))
        self.grad_spans = spans
        for gi, off, a, n in spans:
            self.grads[gi] = self.gbuf[off:off + n]
            self.grad_lo[gi] = a
            ptrs[gi] = self.grads[gi].data_ptr() - 2 * a
        gaps = E - covered  # alignment gaps between members: padding, zeroed by the pack
        self.bytes["pads"] += gaps
        self.bytes["pack"] += 2 * gaps
        self.bytes["total"] += 2 * gaps
        self.gptrs = torch.from_numpy(ptrs).to(dev)
        self.hp = bq.adam_hparams(cfg.lr, cfg.b1, cfg.b2, cfg.eps, cfg.t)
        self.kinds = sorted(kinds)
        self.launches = 1 + len(kinds)
        self.unit_S = {u.name: T.S for u, T in zip(cfg.units, tables)}
        torch.cuda.synchronize(dev)

    def pack(self, stream, gptrs=None, accumulate=False):
        self.bq.pack(self.shard, self.gptrs if gptrs is None else gptrs, self.dbuf, 1.0 / self.V, accumulate,
                     stream=stream)

    def adam(self, stream, fp8=None, fs=None):
        self.bq.step_adam8(self.shard, self.dbuf, self.master, self.m, self.v, self.ms, self.vs, self.hp,
                           self.fp8 if fp8 is None else fp8, self.fs if fs is None else fs, stream=stream)

    def step(self, stream):
        self.pack(stream)
        self.adam(stream)

    def describe(self):
        c = self.cfg
        units = ", ".join(f"{u.name} x{u.repeat}" if u.repeat > 1 else u.name for u in c.units)
        return (f"{self.name}: local shard{'s' if self.hi - self.lo > 1 else ''} {self.lo}..{self.hi - 1} of V={self.V} "
                f"of every unit ({units}; {len(self.members)} members) in one group")


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
        # one pinned host buffer with every gradient at its offset in the
        # device's gradient allocation: one upload per step
        self.host_grads = torch.empty(step.gbuf.numel(), dtype=torch.bfloat16, pin_memory=True)
        self.host_grads.copy_(step.gbuf)
        self.host_fp8 = torch.empty(step.fp8.numel(), dtype=torch.uint8, pin_memory=True)
        self.host_fs = torch.empty(step.fs.numel(), dtype=torch.float32, pin_memory=True)
        self.h2d = step.gbuf.numel() * 2
        self.d2h = step.fp8.numel() + step.fs.numel() * 4
        second = torch.empty_like(step.gbuf)
        ptrs = np.zeros(len(step.gptrs), np.int64)
        for gi, off, a, n in step.grad_spans:
            ptrs[gi] = second[off:off + n].data_ptr() - 2 * a
        self.gbufs = [step.gbuf, second]
        self.gptrs = [step.gptrs, torch.from_numpy(ptrs).to(dev)]
        self.fp8 = [step.fp8, torch.empty_like(step.fp8)]
        self.fs = [step.fs, torch.empty_like(step.fs)]
        self.up, self.down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]  # noqa: E731
        self.ev_up, self.ev_packed, self.ev_adam, self.ev_down = ev(), ev(), ev(), ev()
        self.k = 0

    def issue(self, comp):
        st, torch, j = self.step, self.torch, self.k & 1
        self.up.wait_event(self.ev_packed[j])  # the pack two steps back has read this set
        with torch.cuda.stream(self.up):
            self.gbufs[j].copy_(self.host_grads, non_blocking=True)
            self.ev_up[j].record(self.up)
        comp.wait_event(self.ev_up[j])
        st.pack(comp, gptrs=self.gptrs[j])
        self.ev_packed[j].record(comp)
        comp.wait_event(self.ev_down[j])  # the read-back two steps back is done with this output
        st.adam(comp, fp8=self.fp8[j], fs=self.fs[j])
        self.ev_adam[j].record(comp)
        self.down.wait_event(self.ev_adam[j])
        with torch.cuda.stream(self.down):
            self.host_fp8.copy_(self.fp8[j], non_blocking=True)
            self.host_fs.copy_(self.fs[j], non_blocking=True)
            self.ev_down[j].record(self.down)
        self.k += 1

    def link(self, comp, reps=3):
        """The host link on this machine, each direction alone: the step's upload and
        its read-back as single copies (best of reps), in ms."""
        torch = self.torch
        best = [float("inf"), float("inf")]
        for _ in range(reps):
            for k, (dst, src) in enumerate(((self.gbufs[0], self.host_grads), (self.host_fp8, self.fp8[0]))):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(comp)
                with torch.cuda.stream(comp):
                    dst.copy_(src, non_blocking=True)
                e1.record(comp)
                torch.cuda.synchronize()
                best[k] = min(best[k], e0.elapsed_time(e1))
        return best

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


def _oracle_slice(arg):
    """One device's slice of one unit through the oracle as it stands (pack,
    8-bit Adam, FP8) on the workload's own seeded inputs (the workloads
    generators); only the oracle calls are timed.  Returns (algorithmic bytes,
    elements, seconds)."""
    name, unit_index, dev, reps = arg
    from oracle import adam8 as OA
    from oracle import fp8 as OF
    from oracle import pack as OP
    from oracle import planner as OPl

    cfg = W.config(name)
    unit = cfg.units[unit_index]
    L = OPl.plan([OPl.TensorDesc(t.rows, t.cols, t.g, t.adam_kind, t.fp8) for t in unit.tensors], cfg.V, cfg.alpha,
                 cfg.start_align)
    T = W.Table(L.export())
    lo, hi, cid = dev, dev + 1, cfg.cfg_id
    grads = {}
    for i in range(T.N):
        a, b = T.owned_range(i, lo, hi)
        if b > a:
            grads[i] = (W.grad_bits(cid, unit_index, i, a, b), a)
    master = W.scatter_local(T, lo, hi, lambda i, a, b: W.master_values(cid, unit_index, i, a, b), np.float32)
    m = W.scatter_local(T, lo, hi, lambda i, a, b: W.mcode_values(cid, unit_index, i, a, b), np.int8)
    v = W.scatter_local(T, lo, hi, lambda i, a, b: W.vcode_values(cid, unit_index, i, a, b), np.uint8)
    m0, m1 = T.slot_range(lo, hi)
    f0, f1 = T.slot_range(lo, hi, fp8=True)
    ms = W.scale_values(cid, unit_index, "m", m0, m1)
    vs = W.scale_values(cid, unit_index, "v", m0, m1)
    n = (hi - lo) * T.S
    dbuf0, fp80, fs0 = np.zeros(n, np.uint16), np.zeros(n, np.uint8), np.zeros(max(f1 - f0, 1), np.float32)
    hp = OA.adam_hparams(cfg.lr, cfg.b1, cfg.b2, cfg.eps, cfg.t)
    spent = 0.0
    for _ in range(reps):
        t0 = time.perf_counter()
        dbuf = OP.pack(L, lo, hi, grads, dbuf0, np.float32(1.0 / cfg.V), False)
        p1 = OA.adam8_step(L, lo, hi, dbuf, master, m, v, ms, vs, hp)[0]
        OF.quant_fp8(L, lo, hi, p1, fp80, fs0)
        spent += time.perf_counter() - t0
    b = step_bytes(T, lo, hi)
    return reps * b["total"], reps * b["elems"], spent


def cpu_info():
    model = platform.processor() or platform.machine()
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    aff = sorted(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else list(range(os.cpu_count() or 1))
    return dict(cpu_model=model, cpu_count=os.cpu_count(), affinity=f"{len(aff)} cpus ({aff[0]}-{aff[-1]})")


def sample_unit(workload):
    """The unit of a workload the CPU legs sample: its repeated layer unit, else its first."""
    units = W.config(workload).units
    return max(range(len(units)), key=lambda u: (units[u].repeat, -u))


def cpu_baseline(workload=WORKLOAD, single_seconds=8.0):
    """The oracle as it stands, timed on the host cores on a bounded sample of the
    benchmarked workload: its layer unit's slice on one device (for the
    Llama-3-70B slice 13.6 M elements, its own seeded inputs), through the
    oracle's pack, 8-bit Adam and FP8.  Two legs: one core, the slice repeated
    for about single_seconds; all cores, one slice per worker process (spawned;
    workers independent, as the blocks are), aggregate = sum of the workers'
    rates."""
    import multiprocessing as mp

    info = cpu_info()
    u = sample_unit(workload)
    cfg = W.config(workload)
    V, d0 = cfg.V, cfg.dev_lo
    b, e, t = _oracle_slice((workload, u, d0, 1))
    reps = max(1, int(round(single_seconds / max(t, 1e-3))) - 1)
    b2, e2, t2 = _oracle_slice((workload, u, d0, reps)) if reps > 0 else (0, 0, 0.0)
    one = (b + b2) / (t + t2) / 1e9
    n1 = 1 + reps
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_slice, [(workload, u, k % V, 1) for k in range(cores)])
    wall = time.perf_counter() - t0
    agg = sum(bb / tt for bb, _, tt in res) / 1e9
    return {"value": round(agg, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"the {workload} {cfg.units[u].name} unit's slice on one device of V={V} ({e} elements, "
                      f"seeded workload inputs): oracle pack + 8-bit Adam + FP8, numpy; {cores} spawned worker "
                      f"processes, one slice each (devices 0..{min(cores, V) - 1}), aggregate of the workers' "
                      f"rates ({wall:.1f} s wall with input generation)",
            "single_core": {"value": round(one, 4), "unit": "GB/s", "cores": 1,
                            "sample": f"the same slice {n1} times on one core ({t + t2:.1f} s of oracle time)"},
            **info}


def cpu_baseline_muon(n=4096, steps=5, seed=5):
    """The oracle's Newton-Schulz (fp64 numpy, the BLAS library's own threads over
    the host cores) on a bounded sample of the batch: its n x n matrix, `steps`
    iterations, seeded N(0, 1e-3) entries.  TFLOP/s on the nominal count."""
    from oracle import muon as OM

    x = np.random.default_rng(seed).standard_normal((n, n)) * 1e-3
    t0 = time.perf_counter()
    OM.newton_schulz(x, steps=steps)
    dt = time.perf_counter() - t0
    flops = steps * OM.ns_cost(n, n)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    return {"value": round(flops / dt / 1e12, 4), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"the batch's {n}x{n} matrix, {steps} Newton-Schulz steps in fp64 numpy (BLAS threads over "
                      f"the host cores), {dt:.1f} s; nominal 4 m^2 n + 2 m^3 per step"}


def time_group(step, stream, steps, warmup):
    """Mean pack and Adam milliseconds of a GroupStep (CUDA events)."""
    import torch

    for _ in range(warmup):
        step.step(stream)
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


def graph_ms(step, stream, steps=10, warmup=3):
    """Milliseconds of one DBuffer step of a GroupStep replayed as a CUDA graph
    (captured around the same C-ABI calls)."""
    import torch

    step.step(stream)  # first launches set kernel attributes outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step.step(stream)
    ms = time_call(g.replay, stream, steps, warmup)
    step.bq.shard_check(step.shard, stream=stream)
    del g
    return ms


def gbs(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)  # before the process group, so NCCL binds each rank to its own GPU
    if world > 1:
        dist.init_process_group("nccl")
    import block_quant_gb300 as bq

    bq.load()
    cfg = W.config(args.workload)
    # rank r steps device r's shard of every unit of a one-device slice (weak
    # scaling, no collective); a whole-buffer workload is stepped whole by every rank
    lo = rank % cfg.V if cfg.dev_hi - cfg.dev_lo == 1 else cfg.dev_lo
    step = GroupStep(args.workload, dev, seed=1000 + rank, dev_lo=lo, members=args.members)
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
    bq.shard_check(step.shard, stream=stream)
    if muon:
        bq.muon_ns_check(muon.ws, stream=stream)
    total_ms = t_start.elapsed_time(t_end)
    pack_ms = [e[0].elapsed_time(e[1]) for e in evs]
    adam_ms = [e[1].elapsed_time(e[2]) for e in evs]
    muon_ms = [e[2].elapsed_time(e[3]) for e in evs] if muon else [0.0]
    dbuf_ms = statistics.mean(p + a for p, a in zip(pack_ms, adam_ms))

    # end to end through the public API from pinned host buffers: each step's
    # gradients uploaded, pack + Adam + FP8, the FP8 staging buffer and scales
    # read back; uploads and read-backs overlap the neighbouring steps' kernels
    pipe = E2EPipeline(step, dev)
    # as many steps as the timed region, so that filling and draining the
    # upload / read-back pipeline is spread over the same count
    e2e_ms = pipe.measure(stream, steps=args.steps)
    h2d, d2h = pipe.h2d, pipe.d2h
    link_ms = pipe.link(stream)
    pipe_h2d_bytes, pipe_fp8_bytes = pipe.h2d, pipe.host_fp8.numel()
    del pipe
    torch.cuda.empty_cache()
    muon_e2e = None
    if muon:
        muon.pin_host()
        muon_e2e = muon.measure_e2e(stream, steps=args.steps)

    extra = {}
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        extra["graph"] = max_over_ranks([graph_ms(step, side)], world, device=dev)[0]
    acc_ms = max_over_ranks([time_call(lambda: step.pack(stream, accumulate=True), stream, steps=10, warmup=3)],
                            world, device=dev)[0]
    dq = None
    if args.dequant:
        view = torch.empty(step.n, dtype=torch.bfloat16, device=dev)
        dq = max_over_ranks([time_call(lambda: bq.dequant_fp8(step.shard, step.fp8, step.fs, view, stream=stream),
                                       stream, steps=10, warmup=3)], world, device=dev)[0]
        del view
    head = dict(bytes=step.bytes, launches=step.launches, kinds=step.kinds, S=step.unit_S, n=step.n,
                members=len(step.members), describe=step.describe())
    if args.extras:
        del step
        torch.cuda.empty_cache()
        # the other configurations, each stepped as a group of its own
        for name, key in ((LAYER, "llama3_8b_layer"), (GPTOSS, "gpt_oss_120b_rank0"),
                          ("llama3-8b-layer-tile32", "adam_tile32"), ("toy", "toy_step")):
            if name == args.workload:
                continue
            cfgV = W.config(name).V
            lo = 0 if name in (LAYER, "llama3-8b-layer-tile32", "toy") else rank % cfgV
            st = GroupStep(name, dev, seed=4000 + rank, dev_lo=lo)
            n_ = 200 if name == "toy" else 20
            p_ms, a_ms = time_group(st, stream, steps=n_, warmup=5)
            with torch.cuda.stream(side):
                g_ms = graph_ms(st, side, steps=n_, warmup=5)
            p_ms, a_ms, g_ms = max_over_ranks([p_ms, a_ms, g_ms], world, device=dev)
            extra[key] = (st.describe(), dict(st.bytes), st.launches, st.kinds, p_ms, a_ms, g_ms)
            del st
            torch.cuda.empty_cache()
    mstep = None
    if args.muon_step:
        ms_obj = MuonStep(dev, seed=3000 + rank)
        mstep = max_over_ranks(list(ms_obj.measure(stream, steps=5, warmup=3)), world, device=dev)
    ms_step, dbuf_ms_max, muon_ms_max, e2e_max, muon_e2e_max, adam_max = max_over_ranks(
        [total_ms / args.steps, dbuf_ms, statistics.mean(muon_ms), e2e_ms, muon_e2e or 0.0,
         statistics.mean(adam_ms)], world, device=dev)
    if rank == 0:
        pk = peaks()
        B = head["bytes"]["total"]
        value = job_throughput(B, world, dbuf_ms_max) / 1e9
        adam_gbs = gbs(head["bytes"]["adam"], adam_max)
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(head["describe"], head["bytes"], head["S"], head["n"], head["members"],
                                      bool(muon), world),
            "hbm_frac": round(value / world / pk["hbm"], 4),
            "useful": {"GB/s": round(job_throughput(B - 2 * head["bytes"]["pads"], world, dbuf_ms_max) / 1e9, 1),
                       "bytes": B - 2 * head["bytes"]["pads"],
                       "note": "value without the pack's 2 B zero write per padding element"},
            "dbuffer_ms": round(dbuf_ms_max, 4),
            "pack": {"ms": round(statistics.mean(pack_ms), 4),
                     "GB/s": round(gbs(head["bytes"]["pack"], statistics.mean(pack_ms)), 1),
                     "bytes": head["bytes"]["pack"]},
            "roofline": {"bound": "hbm",
                         "kernel": ROOFLINE_KERNEL[args.workload],
                         "achieved": round(adam_gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                         "frac": round(adam_gbs / pk["hbm"], 4),
                         "traffic": recorded_traffic("bq_step_adam8") if args.workload == WORKLOAD else None,
                         "peak_source": f"{pk['src']} hbm_gbs (STREAM-style copy)",
                         "ms": round(adam_max, 4), "algorithmic_bytes": head["bytes"]["adam"],
                         "launches_per_call": head["launches"] - 1},
            "e2e": {"value": round(job_throughput(B, world, e2e_max) / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "overlap": "upload of step k+1 and read-back of step k run on their own streams during step k",
                    "ms_per_step": round(e2e_max, 4),
                    "link": {"h2d_GB/s": round(gbs(pipe_h2d_bytes, link_ms[0]), 1),
                             "d2h_GB/s": round(gbs(pipe_fp8_bytes, link_ms[1]), 1),
                             "note": "the host link measured on this box after the timed steps, each direction "
                                     "alone (the gradient upload; the FP8 buffer's read-back); both directions "
                                     "at once share it"}},
            "gpu_launches": args.steps * (head["launches"] + (muon_launches(muon) if muon else 0)),
            "clocks": clk,
        }
        if muon:
            tf = job_throughput(muon.flops, world, muon_ms_max) / 1e12
            ex = muon_executed_flops(muon.shapes)
            ex_tf = job_throughput(ex, world, muon_ms_max) / 1e12
            line["muon"] = {"value": round(tf, 1), "unit": "TFLOP/s", "ms": round(muon_ms_max, 3),
                            "flops": muon.flops,
                            "count": "nominal 4 m^2 n + 2 m^3 per step; X X^T and A A^T are computed on "
                                     "the tiles touching the upper triangle only, so this is an effective rate",
                            "executed_flops": ex, "executed_TFLOP/s": round(ex_tf, 1),
                            "frac": round(ex_tf / world / pk["bf16"], 4),
                            "frac_basis": "executed FLOPs (the tiles that run) / measured burst bf16 peak",
                            "frac_sustained": round(ex_tf / world / pk["bf16_sus"], 4),
                            "nominal_over_burst_peak": round(tf / world / pk["bf16"], 4),
                            "peak": pk["bf16"], "peak_sustained": pk["bf16_sus"],
                            "peak_source": f"{pk['src']} bf16_tflops (burst) and bf16_tflops_sustained",
                            "e2e": {"value": round(job_throughput(muon.flops, world, muon_e2e_max) / 1e12, 1),
                                    "unit": "TFLOP/s", "h2d_bytes_per_step": muon.h2d,
                                    "d2h_bytes_per_step": muon.d2h, "ms_per_step": round(muon_e2e_max, 3)}}
        line["dbuffer_graph"] = {
            "ms": round(extra["graph"], 4), "GB/s": round(gbs(B, extra["graph"]), 1),
            "frac": round(gbs(B, extra["graph"]) / pk["hbm"], 4),
            "note": "the same group step replayed as a CUDA graph around the same C-ABI calls; measured after the "
                    "timed region; not part of value"}
        acc_bytes = 6 * head["bytes"]["elems"] + 2 * head["bytes"]["pads"]
        line["pack_accumulate"] = {
            "workload": "the same slice's pack with accumulation (read grad 2 + DBuffer 2, write 2 per element; "
                        "padding zeroed)",
            "ms": round(acc_ms, 4), "GB/s": round(gbs(acc_bytes, acc_ms), 1),
            "frac": round(gbs(acc_bytes, acc_ms) / pk["hbm"], 4), "bytes": acc_bytes,
            "note": "measured after the timed region; not part of value"}
        if dq:
            dq_bytes = 3 * head["bytes"]["fp8_elems"] + 4 * head["bytes"]["fp8_tiles"]
            line["dequant_view"] = {
                "workload": "the same slice's FP8 staging buffer -> bf16 view (code x tile scale)",
                "ms": round(dq, 4), "GB/s": round(gbs(dq_bytes, dq), 1),
                "frac": round(gbs(dq_bytes, dq) / pk["hbm"], 4), "bytes": dq_bytes,
                "note": "measured after the timed region; not part of value"}
        for key in ("llama3_8b_layer", "gpt_oss_120b_rank0", "adam_tile32", "toy_step"):
            if key not in extra:
                continue
            desc, by, ln, kinds, p_ms, a_ms, g_ms = extra[key]
            obj = {"workload": desc, "elements": by["elems"], "bytes": by["total"], "launches": ln,
                   "kernel_families": kinds,
                   "eager": {"ms": round(p_ms + a_ms, 4), "GB/s": round(gbs(by["total"], p_ms + a_ms), 1),
                             "frac": round(gbs(by["total"], p_ms + a_ms) / pk["hbm"], 4)},
                   "pack": {"ms": round(p_ms, 4), "GB/s": round(gbs(by["pack"], p_ms), 1)},
                   "adam": {"ms": round(a_ms, 4), "GB/s": round(gbs(by["adam"], a_ms), 1),
                            "frac": round(gbs(by["adam"], a_ms) / pk["hbm"], 4)},
                   "cuda_graph": {"ms": round(g_ms, 4), "GB/s": round(gbs(by["total"], g_ms), 1),
                                  "frac": round(gbs(by["total"], g_ms) / pk["hbm"], 4)},
                   "note": "measured after the timed region; not part of value"}
            if key == "toy_step":
                obj["note"] = "L2-resident and launch-bound; " + obj["note"]
            line[key] = obj
        if mstep:
            mo, ns, ap = mstep
            tf = ms_obj.flops / (ns * 1e-3) / 1e12
            ex_tf = muon_executed_flops(ms_obj.shapes) / (ns * 1e-3) / 1e12
            gb_m = gbs(12 * ms_obj.elems, mo)
            gb_a = gbs(10 * ms_obj.elems, ap)
            line["muon_step"] = {
                "workload": "llama3-8b-layer, its 7 matrices on Muon (V=8, all shards): momentum + gather, "
                            "Newton-Schulz x 5 on the gathered matrices, apply",
                "ms": round(mo + ns + ap, 3), "muon_elements": ms_obj.elems,
                "momentum": {"ms": round(mo, 4), "GB/s": round(gb_m, 1), "frac": round(gb_m / pk["hbm"], 4),
                             "bytes": 12 * ms_obj.elems},
                "ns": {"ms": round(ns, 3), "TFLOP/s": round(tf, 1), "flops": ms_obj.flops,
                       "count": "nominal (effective: symmetric products run on the upper triangle)",
                       "executed_TFLOP/s": round(ex_tf, 1), "frac": round(ex_tf / pk["bf16"], 4),
                       "frac_sustained": round(ex_tf / pk["bf16_sus"], 4),
                       "frac_basis": "executed FLOPs / measured burst (and sustained) bf16 peak"},
                "apply": {"ms": round(ap, 4), "GB/s": round(gb_a, 1), "frac": round(gb_a / pk["hbm"], 4),
                          "bytes": 10 * ms_obj.elems},
                "root_ns_tflop_per_device": ms_obj.root_tflop,
                "note": "measured after the timed region; not part of value"}
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload)
            if muon:
                line["cpu_baseline"]["muon"] = cpu_baseline_muon()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def muon_launches(muon, steps=5):
    """Kernels one bq_muon_ns call launches: per matrix a sum-of-squares
    reduction, its one-block finish, a scaled (transposing) copy, three GEMMs
    per step and the copy out."""
    return len(muon.mats) * (4 + 3 * steps)


def workload_config(describe, b, S, n, members, muon, world):
    """The config object both arms print (b: step bytes of the benchmarked slice)."""
    return {
        "workload": describe + " + Muon NS batch [4096x4096, 4096x14336, 14336x4096] x 5 iterations" * bool(muon),
        "elements": b["elems"], "padding_elements": b["pads"], "S": S, "members": members,
        "bytes_per_step": b["total"], "l2": f"inputs {n * 13 / 1e9:.1f} GB > L2: no flush needed",
        "launch": "eager: one bq_pack and one bq_step_adam8 call over the whole group per step",
        "parallelism": f"dp{world}: rank r steps device r's shard of every unit, no data-path collective",
    }


def reference_config(args, world):
    """Our arm's config, with the layout figures from the oracle planner (this
    arm runs no library code) and the same member alignment."""
    from oracle import planner as OP

    cfg = W.config(args.workload)
    lo, hi = cfg.dev_lo, cfg.dev_hi
    tot = {k: 0 for k in ("elems", "pads", "pack", "adam", "total", "adam_blocks", "fp8_tiles", "fp8_elems")}
    S, end, covered = {}, 0, 0
    mem = [u for u, unit in enumerate(cfg.units) for _ in range(unit.repeat)]
    if args.members:
        mem = mem[:args.members]
    tabs = {}
    for u in set(mem):
        t = cfg.units[u].tensors
        L = OP.plan([OP.TensorDesc(x.rows, x.cols, x.g, x.adam_kind, x.fp8) for x in t], cfg.V, cfg.alpha,
                    cfg.start_align)
        tabs[u] = W.Table(L.export())
        S[cfg.units[u].name] = tabs[u].S
    for u in mem:
        T = tabs[u]
        end = -(-end // GROUP_ALIGN) * GROUP_ALIGN + (hi - lo) * T.S
        covered += (hi - lo) * T.S
        for k, v in step_bytes(T, lo, hi).items():
            tot[k] += v
    gaps = end - covered
    tot["pads"] += gaps
    tot["pack"] += 2 * gaps
    tot["total"] += 2 * gaps
    units = ", ".join(f"{u.name} x{u.repeat}" if u.repeat > 1 else u.name for u in cfg.units)
    describe = (f"{args.workload}: local shard{'s' if hi - lo > 1 else ''} {lo}..{hi - 1} of V={cfg.V} of every "
                f"unit ({units}; {len(mem)} members) in one group")
    return workload_config(describe, tot, S, end, len(mem), args.muon, world)


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores, same
    metric and unit; each step one device's slice of the 70B layer unit through
    the oracle (a bounded sample of the workload)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    u, d0 = sample_unit(args.workload), W.config(args.workload).dev_lo
    for _ in range(args.warmup):
        _oracle_slice((args.workload, u, d0, 1))
    res = [_oracle_slice((args.workload, u, d0, 1)) for _ in range(args.steps)]
    v = sum(b for b, _, _ in res) / sum(t for _, _, t in res) / 1e9
    ms = 1e3 * statistics.mean(t for _, _, t in res)
    line = {
        "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": reference_config(args, world),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step the {args.workload} {W.config(args.workload).units[u].name} unit's "
                                   f"slice on device {d0} ({res[0][1]} elements, seeded workload inputs) through the "
                                   "oracle's pack, 8-bit Adam and FP8 on one core",
                         **cpu_info()},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--muon", dest="muon", action="store_true", default=True)
    ap.add_argument("--no-muon", dest="muon", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extras", dest="extras", action="store_true", default=True)
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--dequant", dest="dequant", action="store_true", default=True)
    ap.add_argument("--no-dequant", dest="dequant", action="store_false")
    ap.add_argument("--muon-step", dest="muon_step", action="store_true", default=True)
    ap.add_argument("--no-muon-step", dest="muon_step", action="store_false")
    ap.add_argument("--workload", default=WORKLOAD, choices=[WORKLOAD, LAYER, GPTOSS],
                    help="the DBuffer step benchmarked (default: the Llama-3-70B rank-0 slice)")
    ap.add_argument("--members", type=int, default=None,
                    help="step only the first K members of the group (smaller case for profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
