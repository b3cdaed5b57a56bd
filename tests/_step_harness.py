"""Shared set-up for the DBuffer-step parity tests: seeded inputs for one unit of
a configuration (or a hand-made tensor list), the CUDA path through the C ABI,
and the oracle on the same inputs."""

import numpy as np
import torch

import block_quant_gb300 as bq
import workloads as W
from oracle import adam8 as OA
from oracle import fp8 as OF
from oracle import pack as OP
from oracle import planner as P

PAD_F32 = np.float32(1234.5)  # sentinels in padding: must survive the step
PAD_I8, PAD_U8 = np.int8(77), np.uint8(77)
GUARD_BYTES = 1024  # canary tail after every device buffer


class StepCase:
    def __init__(self, cfg, unit_index=0, dev_lo=None, dev_hi=None, tensors=None, V=None, t=None,
                 zero_state=False, zero_tensors=()):
        self.cfg = cfg
        self.unit = cfg.units[unit_index] if tensors is None else W.Unit("custom", tensors)
        self.uid = unit_index
        self.V = cfg.V if V is None else V
        self.dev_lo = cfg.dev_lo if dev_lo is None else dev_lo
        self.dev_hi = cfg.dev_hi if dev_hi is None else dev_hi
        self.t = cfg.t if t is None else t
        descs = [P.TensorDesc(x.rows, x.cols, x.g, x.adam_kind, x.fp8) for x in self.unit.tensors]
        self.olayout = P.plan(descs, self.V, cfg.alpha, cfg.start_align)
        self.layout = bq.plan(self.unit.tensors, self.V, cfg.alpha, cfg.start_align)
        ex = self.layout.export()
        assert np.array_equal(ex, np.asarray(self.olayout.export(), np.int64))
        self.table = W.Table(ex)
        self.S = self.table.S
        self.n = (self.dev_hi - self.dev_lo) * self.S
        m0, m1 = self.table.slot_range(self.dev_lo, self.dev_hi)
        f0, f1 = self.table.slot_range(self.dev_lo, self.dev_hi, fp8=True)
        self.nm, self.nf = m1 - m0, f1 - f0
        cid, uid = cfg.cfg_id, unit_index
        zt = set(zero_tensors)

        def gvals(i, a, b):
            return np.zeros(b - a, np.uint16) if i in zt else W.grad_bits(cid, uid, i, a, b)

        self.grads = {}
        for i in range(len(self.unit.tensors)):
            lo, hi = self.table.owned_range(i, self.dev_lo, self.dev_hi)
            if hi > lo:
                self.grads[i] = (gvals(i, lo, hi), lo)
        T, dl, dh = self.table, self.dev_lo, self.dev_hi
        self.master = W.scatter_local(T, dl, dh, lambda i, a, b: np.zeros(b - a, np.float32) if i in zt
                                      else W.master_values(cid, uid, i, a, b), np.float32, fill=PAD_F32)
        if zero_state:
            self.m = W.scatter_local(T, dl, dh, lambda i, a, b: np.zeros(b - a, np.int8), np.int8, fill=PAD_I8)
            self.v = W.scatter_local(T, dl, dh, lambda i, a, b: np.zeros(b - a, np.uint8), np.uint8, fill=PAD_U8)
            self.ms = np.zeros(self.nm, np.float32)
            self.vs = np.zeros(self.nm, np.float32)
        else:
            self.m = W.scatter_local(T, dl, dh, lambda i, a, b: W.mcode_values(cid, uid, i, a, b), np.int8, fill=PAD_I8)
            self.v = W.scatter_local(T, dl, dh, lambda i, a, b: W.vcode_values(cid, uid, i, a, b), np.uint8, fill=PAD_U8)
            self.ms = W.scale_values(cid, uid, "m", m0, m1)
            self.vs = W.scale_values(cid, uid, "v", m0, m1)
        self.dbuf0 = np.full(self.n, 0x3F80, np.uint16)  # 1.0: pack must overwrite or zero it
        self.fp8_0 = np.full(self.n, 0xAA, np.uint8)
        self.fs0 = np.full(max(self.nf, 1), np.nan, np.float32)
        self.hp_o = OA.adam_hparams(cfg.lr, cfg.b1, cfg.b2, cfg.eps, self.t)
        self.hp_c = bq.adam_hparams(cfg.lr, cfg.b1, cfg.b2, cfg.eps, self.t)

    # ------------------------------------------------------------------ CUDA path
    def run_gpu(self, dev, scale=None, accumulate=False, fp8=True, reps=1):
        # every device buffer gets a canary tail: a write past the end of any
        # output shows up as a changed tail (the sanitizer stand-in)
        guards = []

        def d(a):
            a = np.ascontiguousarray(a)
            tail = np.frombuffer(np.full(GUARD_BYTES, 0x5A, np.uint8).tobytes(), dtype=a.dtype)
            full = torch.from_numpy(np.concatenate([a.reshape(-1), tail])).to(dev)
            guards.append((full, a.size))
            return full[:a.size]

        s = torch.cuda.current_stream(dev)
        ws = torch.empty(self.layout.upload_bytes(self.dev_lo, self.dev_hi), dtype=torch.uint8, device=dev)
        shard = self.layout.upload(self.dev_lo, self.dev_hi, ws, stream=s)
        gbufs, ptrs = [], np.zeros(len(self.unit.tensors), np.int64)
        for i, (bits, lo) in self.grads.items():
            g = d(bits.view(np.int16))
            gbufs.append(g)
            ptrs[i] = g.data_ptr() - 2 * lo
        gp = d(ptrs)
        dbuf = d(self.dbuf0.view(np.int16))
        master, m, v = d(self.master), d(self.m), d(self.v)
        ms, vs = d(self.ms), d(self.vs)
        fp8_out = d(self.fp8_0) if fp8 else None
        fs = d(self.fs0) if fp8 else None
        sc = 1.0 / self.V if scale is None else scale
        for _ in range(reps):
            bq.pack(shard, gp, dbuf, sc, accumulate, stream=s)
            bq.step_adam8(shard, dbuf, master, m, v, ms, vs, self.hp_c, fp8_out, fs, stream=s)
        # standalone requantisation of the updated master into separate buffers
        q2 = d(self.fp8_0)
        s2 = d(self.fs0)
        bq.quant_fp8(shard, master, q2, s2, stream=s)
        bq.shard_check(shard, stream=s)  # no bounded device wait gave up
        torch.cuda.synchronize(dev)
        for full, n in guards:
            tail = full[n:].cpu().numpy().view(np.uint8)
            assert np.all(tail == 0x5A), f"write past the end of a {n}-element buffer"
        h = lambda t: None if t is None else t.cpu().numpy()  # noqa: E731
        out = dict(dbuf=h(dbuf).view(np.uint16), master=h(master), m=h(m), v=h(v), ms=h(ms), vs=h(vs),
                   fp8=h(fp8_out), fs=h(fs), q2=h(q2), s2=h(s2))
        del gbufs
        return out

    # ------------------------------------------------------------------ oracle
    def run_oracle(self, scale=None, accumulate=False, blocks=None, tiles=None):
        sc = np.float32(1.0 / self.V if scale is None else scale)
        L, lo, hi = self.olayout, self.dev_lo, self.dev_hi
        dbuf = OP.pack(L, lo, hi, self.grads, self.dbuf0, sc, accumulate)
        master, m, v, ms, vs = OA.adam8_step(L, lo, hi, dbuf, self.master, self.m, self.v, self.ms, self.vs,
                                             self.hp_o, blocks=blocks)
        q, fs = OF.quant_fp8(L, lo, hi, master, self.fp8_0, self.fs0, tiles=tiles)
        return dict(dbuf=dbuf, master=master, m=m, v=v, ms=ms, vs=vs, fp8=q, fs=fs)


def assert_bits_equal(name, got, want):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    if got.dtype.kind == "f":
        gb, wb = got.view(np.uint32 if got.itemsize == 4 else np.uint64), want.view(np.uint32 if want.itemsize == 4 else np.uint64)
    else:
        gb, wb = got, want
    bad = np.nonzero(gb != wb)[0]
    assert bad.size == 0, f"{name}: {bad.size} of {got.size} differ, first at {bad[:8]}: got {got[bad[:4]]} want {want[bad[:4]]}"


def sampled_check(case, got, n_blocks=300, n_tiles=24, seed=0):
    """Full-size parity on sampled outputs: the whole packed gradient buffer is
    compared with the oracle's pack; Adam blocks and FP8 tiles holding random
    tensor elements are recomputed by the oracle one by one; padding of every
    state buffer must be untouched."""
    from oracle import adam8 as OA
    from oracle import fp8 as OF
    from oracle import pack as OP
    from oracle import planner as P

    L, lo, hi = case.olayout, case.dev_lo, case.dev_hi
    sc = np.float32(1.0 / case.V)
    dbuf = OP.pack(L, lo, hi, case.grads, case.dbuf0, sc, False)
    assert_bits_equal("dbuf (full)", got["dbuf"], dbuf)
    covered = np.zeros(case.n, bool)
    for k, i, t_off, ln, loff, _, _ in L.intervals[L.dev_table[lo][0]:L.dev_table[hi][0]]:
        covered[(k - lo) * L.S + loff:(k - lo) * L.S + loff + ln] = True
    assert np.all(got["master"][~covered] == PAD_F32) and np.all(got["m"][~covered] == PAD_I8)
    assert np.all(got["v"][~covered] == PAD_U8)
    rng = np.random.default_rng(seed)

    def probes(count):
        """random tensor positions (padding rejected), with replacement"""
        out = []
        while len(out) < count:
            cand = rng.integers(0, case.n, size=4 * count)
            out.extend(int(x) for x in cand[covered[cand]])
        return out[:count]

    p_new = {}

    def run_block(slot, pos):
        p1, qm, qv, sm, sv = OA.adam8_block(dbuf[pos], case.master[pos], case.m[pos], case.v[pos],
                                            case.ms[slot], case.vs[slot], case.hp_o)
        p_new.update(zip(pos.tolist(), p1.tolist()))
        return p1, qm, qv, sm, sv

    for probe in probes(n_blocks):
        slot, pos = P.block_at(L, lo, hi, probe)
        p1, qm, qv, sm, sv = run_block(slot, pos)
        assert_bits_equal(f"master block {slot}", got["master"][pos], p1)
        assert_bits_equal(f"m codes block {slot}", got["m"][pos], qm)
        assert_bits_equal(f"v codes block {slot}", got["v"][pos], qv)
        assert_bits_equal(f"m scale {slot}", got["ms"][slot:slot + 1], np.array([sm], np.float32))
        assert_bits_equal(f"v scale {slot}", got["vs"][slot:slot + 1], np.array([sv], np.float32))
    if got["fp8"] is None:
        return
    if case.nf == 0:  # no FP8 tiles in the range: the staging buffer is untouched
        assert np.all(got["fp8"] == case.fp8_0)
        return
    done = 0
    for probe in probes(20 * n_tiles):
        if done >= n_tiles:
            break
        hit = P.block_at(L, lo, hi, probe, fp8=True)
        if hit is None:
            continue
        tslot, tpos = hit
        # every Adam block meeting the tile: blocks are at least 128 elements
        # long and tile rows are 8-element aligned, so probing every 8th
        # element finds them all
        need = set()
        for e in np.unique(np.concatenate([tpos[::8], tpos[7::8]])):
            need.add(int(e))
        for e in sorted(need):
            if e not in p_new:
                slot, pos = P.block_at(L, lo, hi, e)
                run_block(slot, pos)
        p_tile = np.array([p_new[int(e)] for e in tpos], np.float32)
        q, s = OF.fp8_tile(p_tile)
        assert_bits_equal(f"fp8 codes tile {tslot}", got["fp8"][tpos], q)
        assert_bits_equal(f"fp8 scale tile {tslot}", got["fs"][tslot:tslot + 1], np.array([s], np.float32))
        assert_bits_equal(f"fp8 codes tile {tslot} (standalone)", got["q2"][tpos], q)
        done += 1
    assert done > 0
