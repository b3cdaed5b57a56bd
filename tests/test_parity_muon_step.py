"""Parity of the Muon step around Newton-Schulz on the GPU, through the C ABI,
against the oracle: momentum + gather and apply bit for bit (the gather also
split over two shard ranges, as two roots' inputs would be); the whole chain
(momentum, Newton-Schulz on the gathered matrices, apply) within the
Newton-Schulz tolerance of the fp64 oracle; full-size sampled checks on the
Llama-3-8B layer with its matrices on Muon."""

import numpy as np
import pytest
import torch

import block_quant_gb300 as bq
import workloads as W
from _step_harness import assert_bits_equal
from oracle import codecs as OC
from oracle import muon as OM
from oracle import pack as OP
from oracle import planner as P

pytestmark = pytest.mark.gpu

PAD_F32 = np.float32(1234.5)
SENT16 = np.uint16(0xFFFF)  # a NaN pattern: never produced by the momentum step here


class MuonCase:
    """Seeded inputs of one unit of a Muon-step configuration over local shards
    [lo, hi): the packed gradient DBuffer (oracle pack of the generator's
    gradients, scale 1/V), prior momentum, master and stand-in NS outputs."""

    def __init__(self, name, lo=None, hi=None):
        cfg = self.cfg = W.config(name)
        self.unit = cfg.units[0]
        self.descs = [P.TensorDesc(t.rows, t.cols, t.g, t.adam_kind, t.fp8) for t in self.unit.tensors]
        self.L = P.plan(self.descs, cfg.V, cfg.alpha, cfg.start_align)
        self.layout = bq.plan(self.unit.tensors, cfg.V, cfg.alpha, cfg.start_align)
        assert np.array_equal(self.layout.export(), np.asarray(self.L.export(), np.int64))
        self.table = W.Table(self.layout.export())
        self.lo = cfg.dev_lo if lo is None else lo
        self.hi = cfg.dev_hi if hi is None else hi
        self.S = self.table.S
        self.n = (self.hi - self.lo) * self.S
        self.muon = [i for i, d in enumerate(self.descs) if d.adam_kind == P.OPT_MUON]
        cid = cfg.cfg_id
        T, lo_, hi_ = self.table, self.lo, self.hi
        grads = {}
        for i in range(len(self.descs)):
            a, b = T.owned_range(i, lo_, hi_)
            if b > a:
                grads[i] = (W.grad_bits(cid, 0, i, a, b), a)
        self.dbuf = OP.pack(self.L, lo_, hi_, grads, np.zeros(self.n, np.uint16), np.float32(1.0 / cfg.V), False)
        self.mom = W.scatter_local(T, lo_, hi_, lambda i, a, b: W.mom_values(cid, 0, i, a, b), np.float32,
                                   fill=PAD_F32)
        self.master = W.scatter_local(T, lo_, hi_, lambda i, a, b: W.master_values(cid, 0, i, a, b), np.float32,
                                      fill=PAD_F32)
        self.lr = np.array([cfg.muon_lr * (1 + 0.125 * i) for i in range(len(self.descs))], np.float32)

    def shard(self, dev):
        ws = torch.empty(self.layout.upload_bytes(self.lo, self.hi), dtype=torch.uint8, device=dev)
        return self.layout.upload(self.lo, self.hi, ws), ws

    def gather_buffers(self, dev):
        bufs = {i: torch.full((self.descs[i].numel,), -1, dtype=torch.int16, device=dev) for i in self.muon}
        ptrs = np.zeros(len(self.descs), np.int64)
        for i, t in bufs.items():
            ptrs[i] = t.data_ptr()
        return bufs, torch.from_numpy(ptrs).to(dev)


def _dev():
    return torch.device("cuda:0")


def _to(dev, a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _pieces_of(case, i):
    return [(pos, t_off, ln) for pos, j, t_off, ln in OM._muon_pieces(case.L, case.lo, case.hi) if j == i]


@pytest.mark.parametrize("name,lo,hi", [("muon-step-small", None, None), ("muon-step-small", 2, 5),
                                        ("muon-step-small", 7, 8)])
def test_momentum_and_gather_bit_exact(cuda, name, lo, hi):
    c = MuonCase(name, lo, hi)
    dev = _dev()
    shard, ws = c.shard(dev)
    mom = _to(dev, c.mom)
    bufs, ptrs = c.gather_buffers(dev)
    bq.muon_momentum(shard, _to(dev, c.dbuf.view(np.int16)), mom, c.cfg.mu, ptrs)
    bq.shard_check(shard)
    want_mom, pieces = OM.muon_momentum(c.L, c.lo, c.hi, c.dbuf, c.mom, c.cfg.mu)
    assert_bits_equal("momentum", mom.cpu().numpy(), want_mom)
    for i in c.muon:
        got = bufs[i].cpu().numpy().view(np.uint16)
        want = np.full(c.descs[i].numel, SENT16, np.uint16)
        for t_off, bits in pieces.get(i, []):
            want[t_off:t_off + len(bits)] = bits
        assert_bits_equal(f"gathered tensor {i}", got, want)


def test_gather_split_over_two_shard_ranges(cuda):
    """Shards [0, 3) and [3, 8) gather into the same matrices, each its owned
    part: together the full matrices, equal to the oracle's assembly."""
    dev = _dev()
    a, b = MuonCase("muon-step-small", 0, 3), MuonCase("muon-step-small", 3, 8)
    bufs, ptrs = a.gather_buffers(dev)
    for c in (a, b):
        shard, ws = c.shard(dev)
        bq.muon_momentum(shard, _to(dev, c.dbuf.view(np.int16)), _to(dev, c.mom), c.cfg.mu, ptrs)
        bq.shard_check(shard)
    _, pa = OM.muon_momentum(a.L, 0, 3, a.dbuf, a.mom, a.cfg.mu)
    _, pb = OM.muon_momentum(b.L, 3, 8, b.dbuf, b.mom, b.cfg.mu)
    for i in a.muon:
        want = OM.assemble(a.descs[i], pa.get(i, []) + pb.get(i, [])).reshape(-1)
        assert_bits_equal(f"assembled tensor {i}", bufs[i].cpu().numpy().view(np.uint16), want)


@pytest.mark.parametrize("lo,hi", [(0, 8), (1, 6)])
def test_apply_bit_exact(cuda, lo, hi):
    c = MuonCase("muon-step-small", lo, hi)
    dev = _dev()
    shard, ws = c.shard(dev)
    ups = {i: W.ns_out_bits(c.cfg.cfg_id, i, c.descs[i].numel) for i in c.muon}
    skip = c.muon[1]  # a NULL pointer skips its tensor
    ups_d = {i: _to(dev, u.view(np.int16)) for i, u in ups.items()}
    ptrs = np.zeros(len(c.descs), np.int64)
    for i, t in ups_d.items():
        ptrs[i] = 0 if i == skip else t.data_ptr()
    master = _to(dev, c.master)
    bq.muon_apply(shard, master, _to(dev, ptrs), _to(dev, c.lr))
    bq.shard_check(shard)
    want = OM.muon_apply(c.L, lo, hi, c.master, {i: u for i, u in ups.items() if i != skip},
                         {i: float(c.lr[i]) for i in c.muon})
    assert_bits_equal("master", master.cpu().numpy(), want)


def test_chain_momentum_ns_apply_within_tolerance(cuda):
    """momentum -> gathered matrices -> Newton-Schulz (tensor cores) -> apply:
    the weight change of every Muon tensor within 2e-2 relative Frobenius of
    -lr * NS64(M) from the oracle's fp64 Newton-Schulz of the same bf16 M."""
    c = MuonCase("muon-step-small")
    dev = _dev()
    shard, ws = c.shard(dev)
    bufs, gptrs = c.gather_buffers(dev)
    bq.muon_momentum(shard, _to(dev, c.dbuf.view(np.int16)), _to(dev, c.mom), c.cfg.mu, gptrs)
    outs = {i: torch.empty_like(bufs[i]) for i in c.muon}
    mats = [(bufs[i].view(torch.bfloat16).view(c.descs[i].rows, c.descs[i].cols),
             outs[i].view(torch.bfloat16).view(c.descs[i].rows, c.descs[i].cols),
             c.descs[i].rows, c.descs[i].cols) for i in c.muon]
    wsn = torch.empty(bq.muon_ns_workspace(mats), dtype=torch.uint8, device=dev)
    bq.muon_ns(mats, wsn, steps=5)
    bq.muon_ns_check(wsn)
    optrs = np.zeros(len(c.descs), np.int64)
    for i in c.muon:
        optrs[i] = outs[i].data_ptr()
    master = _to(dev, c.master)
    bq.muon_apply(shard, master, _to(dev, optrs), _to(dev, c.lr))
    bq.shard_check(shard)
    w1 = master.cpu().numpy().astype(np.float64)
    _, pieces = OM.muon_momentum(c.L, c.lo, c.hi, c.dbuf, c.mom, c.cfg.mu)
    for i in c.muon:
        m_bits = OM.assemble(c.descs[i], pieces[i])
        assert_bits_equal(f"NS input {i}", bufs[i].cpu().numpy().view(np.uint16), m_bits.reshape(-1))
        o64 = OM.newton_schulz(OC.bf16_bits_to_f32(m_bits)).reshape(-1)
        got, want = [], []
        for pos, t_off, ln in _pieces_of(c, i):
            got.append(w1[pos:pos + ln] - c.master[pos:pos + ln].astype(np.float64))
            want.append(-float(c.lr[i]) * o64[t_off:t_off + ln])
        got, want = np.concatenate(got), np.concatenate(want)
        err = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert err <= 2e-2, (i, err)
    # non-Muon tensors and padding untouched
    muon = np.zeros(c.n, bool)
    for pos, _, _, ln in OM._muon_pieces(c.L, c.lo, c.hi):
        muon[pos:pos + ln] = True
    assert np.array_equal(w1[~muon].astype(np.float32), c.master[~muon])


def test_full_size_sampled(cuda):
    """Llama-3-8B layer, matrices on Muon, all 8 shards (218 M parameters):
    momentum, gather and apply checked at sampled positions against the oracle's
    element formulas; elements of other tensors and padding untouched."""
    cfg = W.config("llama3-8b-layer-muon")
    unit = cfg.units[0]
    descs = [P.TensorDesc(t.rows, t.cols, t.g, t.adam_kind, t.fp8) for t in unit.tensors]
    layout = bq.plan(unit.tensors, cfg.V, cfg.alpha, cfg.start_align)
    L = P.plan(descs, cfg.V, cfg.alpha, cfg.start_align)
    assert np.array_equal(layout.export(), np.asarray(L.export(), np.int64))
    T = W.Table(layout.export())
    lo, hi, S = 0, cfg.V, T.S
    n = (hi - lo) * S
    dev = _dev()
    ws = torch.empty(layout.upload_bytes(lo, hi), dtype=torch.uint8, device=dev)
    shard = layout.upload(lo, hi, ws)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    dbuf = (torch.randn(n, generator=g, device=dev) * 1e-3).to(torch.bfloat16)
    mom0 = torch.randn(n, generator=g, device=dev) * 1e-3
    w0 = torch.randn(n, generator=g, device=dev) * 0.02
    muon = [i for i, d in enumerate(descs) if d.adam_kind == P.OPT_MUON]
    gath = {i: torch.zeros(descs[i].numel, dtype=torch.bfloat16, device=dev) for i in muon}
    ups = {i: (torch.randn(descs[i].numel, generator=g, device=dev) * 0.02).to(torch.bfloat16) for i in muon}
    gp, up = np.zeros(len(descs), np.int64), np.zeros(len(descs), np.int64)
    for i in muon:
        gp[i], up[i] = gath[i].data_ptr(), ups[i].data_ptr()
    lr = torch.from_numpy(np.array([cfg.muon_lr * (1 + 0.125 * i) for i in range(len(descs))], np.float32)).to(dev)
    mom, w = mom0.clone(), w0.clone()
    bq.muon_momentum(shard, dbuf, mom, cfg.mu, torch.from_numpy(gp).to(dev))
    bq.muon_apply(shard, w, torch.from_numpy(up).to(dev), lr)
    bq.shard_check(shard)
    pieces = list(OM._muon_pieces(L, lo, hi))
    muon_mask = torch.zeros(n, dtype=torch.bool, device=dev)
    for pos, _, _, ln in pieces:
        muon_mask[pos:pos + ln] = True
    assert torch.equal(mom[~muon_mask], mom0[~muon_mask]) and torch.equal(w[~muon_mask], w0[~muon_mask])
    rng = np.random.default_rng(0)
    for pos, i, t_off, ln in pieces:
        j = np.unique(np.concatenate([rng.integers(0, ln, 4096), [0, ln - 1]]))
        p = torch.from_numpy(pos + j).to(dev)
        g_bits = dbuf[p].view(torch.int16).cpu().numpy().view(np.uint16)
        m_prev, m_new = mom0[p].cpu().numpy(), mom[p].cpu().numpy()
        want_m = OC.fma32(np.full(j.size, np.float32(cfg.mu)), m_prev, OC.bf16_bits_to_f32(g_bits))
        assert_bits_equal(f"momentum tensor {i}", m_new, want_m)
        toff = torch.from_numpy(t_off + j).to(dev)
        assert_bits_equal(f"gathered tensor {i}", gath[i][toff].view(torch.int16).cpu().numpy().view(np.uint16),
                          OC.f32_to_bf16_bits(want_m))
        o = OC.bf16_bits_to_f32(ups[i][toff].view(torch.int16).cpu().numpy().view(np.uint16))
        want_w = OC.fma32(np.full(j.size, -np.float32(lr[i].item())), o, w0[p].cpu().numpy())
        assert_bits_equal(f"master tensor {i}", w[p].cpu().numpy(), want_w)
