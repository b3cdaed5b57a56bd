"""Pins of the oracle's pack, 8-bit Adam, FP8 and Newton-Schulz steps against
round trips, closed forms and library routines (no GPU)."""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import adam8 as A
from oracle import codecs as C
from oracle import fp8 as F
from oracle import muon as M
from oracle import pack as PK
from oracle import planner as P


def _layout(name):
    c = W.config(name)
    u = c.units[0]
    d = [P.TensorDesc(t.rows, t.cols, t.g, t.adam_kind, t.fp8) for t in u.tensors]
    return c, u, P.plan(d, c.V, c.alpha, c.start_align)


def _grads(c, u, L, dev_lo, dev_hi):
    t = W.Table(L.export())
    out = {}
    for i in range(len(u.tensors)):
        lo, hi = t.owned_range(i, dev_lo, dev_hi)
        if hi > lo:
            out[i] = (W.grad_bits(c.cfg_id, 0, i, lo, hi), lo)
    return out


# ----------------------------------------------------------------------------- pack


@pytest.mark.parametrize("name,dev", [("gptoss-small", (0, 8)), ("llama-small", (2, 5)), ("toy", (3, 4))])
def test_pack_unpack_roundtrip(name, dev):
    c, u, L = _layout(name)
    lo, hi = dev
    grads = _grads(c, u, L, lo, hi)
    junk = np.full((hi - lo) * L.S, 0x3F80, np.uint16)  # 1.0 everywhere beforehand
    out = PK.pack(L, lo, hi, grads, junk, 1.0, False)
    back = PK.unpack(L, lo, hi, out)
    assert set(back) == set(grads)
    for i, (bits, base) in grads.items():
        assert back[i][1] == base and np.array_equal(back[i][0], bits)
    # padding zeroed, tensor elements untouched by scale 1
    covered = np.zeros(out.size, bool)
    for (k, i, t_off, ln, loff, _, _) in L.intervals[L.dev_table[lo][0]:L.dev_table[hi][0]]:
        covered[(k - lo) * L.S + loff:(k - lo) * L.S + loff + ln] = True
    assert not out[~covered].any()
    # sum preserved (scale 1)
    tot_in = sum(C.bf16_bits_to_f32(b).astype(np.float64).sum() for b, _ in grads.values())
    assert np.isclose(C.bf16_bits_to_f32(out).astype(np.float64).sum(), tot_in, rtol=0, atol=1e-9)


def test_pack_scale_and_accumulate():
    c, u, L = _layout("llama-small")
    grads = _grads(c, u, L, 0, c.V)
    zero = np.zeros(c.V * L.S, np.uint16)
    once = PK.pack(L, 0, c.V, grads, zero, 1.0, False)
    eighth = PK.pack(L, 0, c.V, grads, zero, 1.0 / 8, False)
    # a power-of-two scale is exact: eighth * 8 == once
    assert np.array_equal(C.f32_to_bf16_bits(C.bf16_bits_to_f32(eighth) * np.float32(8)), once)
    twice = PK.pack(L, 0, c.V, grads, once, 1.0, True)
    assert np.array_equal(C.f32_to_bf16_bits(C.bf16_bits_to_f32(once) * np.float32(2)), twice)
    # general scale / accumulate against torch's own bf16 arithmetic
    sc = 0.3
    acc = PK.pack(L, 0, c.V, grads, twice, sc, True)
    for (k, i, t_off, ln, loff, _, _) in L.intervals:
        pos = k * L.S + loff
        src = torch.from_numpy(grads[i][0][t_off - grads[i][1]:][:ln].view(np.int16)).view(torch.bfloat16).float()
        dst = torch.from_numpy(twice[pos:pos + ln].view(np.int16)).view(torch.bfloat16).float()
        want = (dst + src * torch.tensor(sc, dtype=torch.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(acc[pos:pos + ln], want)


# ----------------------------------------------------------------------------- Adam


HP = dict(lr=1e-3, b1=0.9, b2=0.999, eps=1e-8)


def test_adam_hparams():
    hp = A.adam_hparams(t=10, **HP)
    assert hp["rbc1"] == np.float32(1 / (1 - 0.9 ** 10)) and hp["omb2"] == np.float32(0.001)
    assert all(v.dtype == np.float32 for v in hp.values())


def test_adam8_first_step_closed_form():
    """t = 1 from zero state: m' = (1-b1) g, v' = (1-b2) g^2, so the step is
    p - lr * g / (|g| + eps) up to fp32 rounding."""
    rng = np.random.default_rng(0)
    g = C.f32_to_bf16_bits((rng.standard_normal(4096) * 1e-3).astype(np.float32))
    p = (rng.standard_normal(4096) * 0.02).astype(np.float32)
    hp = A.adam_hparams(t=1, **HP)
    p1, qm, qv, sm, sv = A.adam8_block(g, p, np.zeros(4096, np.int8), np.zeros(4096, np.uint8),
                                       np.float32(0), np.float32(0), hp)
    gf = C.bf16_bits_to_f32(g).astype(np.float64)
    want = p - 1e-3 * gf / (np.abs(gf) + 1e-8)
    assert np.allclose(p1, want, rtol=1e-6, atol=1e-9)
    assert np.max(np.abs(qm.astype(int))) == 127 and qv.max() == 255
    assert np.isclose(sm, np.max(np.abs(0.1 * gf)) / 127, rtol=1e-6)


def test_adam_update_matches_torch_adam():
    """With quantisation bypassed (state carried in fp32) the update is Adam:
    compare five steps with torch.optim.Adam (CPU, foreach=False)."""
    rng = np.random.default_rng(1)
    n = 3000
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.Adam([tp], lr=HP["lr"], betas=(HP["b1"], HP["b2"]), eps=HP["eps"], foreach=False)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, 6):
        gb = C.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
        tp.grad = torch.from_numpy(C.bf16_bits_to_f32(gb).copy())
        opt.step()
        p, m, v = A.adam_update(gb, p, m, v, A.adam_hparams(t=t, **HP))
        st = opt.state[tp]
        tm, tv = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        # torch forms m by lerp: a few ulps of the largest |m| apart at most
        assert np.allclose(m, tm, rtol=1e-5, atol=1e-6 * np.abs(tm).max())
        assert np.allclose(v, tv, rtol=1e-5, atol=1e-6 * tv.max())
        # different but equally valid fp32 op orders: allow a few ulps of p and
        # 1e-5 of the step size lr
        assert np.allclose(p, tp.detach().numpy(), rtol=1e-6, atol=1e-5 * HP["lr"])


def test_adam8_step_over_layout():
    c, u, L = _layout("gptoss-small")
    t = W.Table(L.export())
    lo, hi = 0, c.V
    grad = W.scatter_local(t, lo, hi, lambda i, a, b: W.grad_bits(c.cfg_id, 0, i, a, b), np.uint16)
    master = W.scatter_local(t, lo, hi, lambda i, a, b: W.master_values(c.cfg_id, 0, i, a, b), np.float32, fill=7.0)
    mq = W.scatter_local(t, lo, hi, lambda i, a, b: W.mcode_values(c.cfg_id, 0, i, a, b), np.int8, fill=5)
    vq = W.scatter_local(t, lo, hi, lambda i, a, b: W.vcode_values(c.cfg_id, 0, i, a, b), np.uint8, fill=5)
    ms = W.scale_values(c.cfg_id, 0, "m", 0, L.n_mslots)
    vs = W.scale_values(c.cfg_id, 0, "v", 0, L.n_mslots)
    hp = A.adam_hparams(t=c.t, lr=c.lr, b1=c.b1, b2=c.b2, eps=c.eps)
    p1, m1, v1, ms1, vs1 = A.adam8_step(L, lo, hi, grad, master, mq, vq, ms, vs, hp)
    pad = master == 7.0
    assert np.array_equal(p1[pad], master[pad]) and np.all(m1[pad] == 5) and np.all(v1[pad] == 5)
    assert np.mean(p1[~pad] != master[~pad]) > 0.99  # a few updates fall below one ulp of p
    for slot, pos in P.adam_blocks(L, lo, hi):
        assert np.max(np.abs(m1[pos].astype(int))) == 127 and np.max(v1[pos]) == 255
        assert ms1[slot] > 0 and vs1[slot] > 0


# ----------------------------------------------------------------------------- FP8


def test_fp8_tile_properties():
    rng = np.random.default_rng(4)
    for n in (1, 77, 128 * 128):
        p = (rng.standard_normal(n) * 0.02).astype(np.float32)
        q, s = F.fp8_tile(p)
        assert s == np.float32(np.max(np.abs(p))) / np.float32(448)
        deq = C.e4m3_decode(q) * np.float64(s)
        assert np.max(np.abs(C.e4m3_decode(q))) == 448.0
        xs = np.abs(p / s).astype(np.float64)
        normal = xs >= 2.0 ** -6
        err = np.abs(deq - p)
        assert np.all(err[normal] <= (2.0 ** -4 + 2.0 ** -22) * np.abs(p[normal]))
        assert np.all(err[~normal] <= (2.0 ** -10 + 2.0 ** -22) * s)


def test_fp8_zero_tile_keeps_sign():
    q, s = F.fp8_tile(np.array([0.0, -0.0, 0.0], np.float32))
    assert s == 0 and list(q) == [0x00, 0x80, 0x00]


def test_quant_fp8_over_layout():
    c, u, L = _layout("llama-tile-small")
    t = W.Table(L.export())
    master = W.scatter_local(t, 0, c.V, lambda i, a, b: W.master_values(c.cfg_id, 0, i, a, b), np.float32)
    out = np.full(c.V * L.S, 0xAA, np.uint8)
    q, s = F.quant_fp8(L, 0, c.V, master, out, np.zeros(L.n_fslots, np.float32))
    for slot, pos in P.fp8_tiles(L, 0, c.V):
        assert s[slot] == np.float32(np.max(np.abs(master[pos]))) / np.float32(448)
        assert np.max(np.abs(C.e4m3_decode(q[pos]))) == 448.0
    covered = np.zeros(out.size, bool)
    for _, pos in P.fp8_tiles(L, 0, c.V):
        covered[pos] = True
    assert np.all(q[~covered] == 0xAA)


# ----------------------------------------------------------------------------- Newton-Schulz


def _phi(x, a=M.NS_A, b=M.NS_B, c=M.NS_C):
    return a * x + b * x ** 3 + c * x ** 5


@pytest.mark.parametrize("shape", [(64, 64), (48, 96), (96, 40), (7, 13)])
def test_newton_schulz_svd_closed_form(shape):
    """NS acts on singular values only: X = U diag(s) V^T maps to
    U diag(phi^5(s / (||s|| + eps))) V^T with phi(x) = a x + b x^3 + c x^5."""
    rng = np.random.default_rng(sum(shape))
    R, Cc = shape
    k = min(R, Cc)
    U, _ = np.linalg.qr(rng.standard_normal((R, k)))
    Vm, _ = np.linalg.qr(rng.standard_normal((Cc, k)))
    s = rng.uniform(0.01, 1.0, k) * 1e-2
    X = U @ np.diag(s) @ Vm.T
    y = M.newton_schulz(X)
    x = s / (np.sqrt(np.sum(s ** 2)) + 1e-7)
    for _ in range(5):
        x = _phi(x)
    want = U @ np.diag(x) @ Vm.T
    assert np.linalg.norm(y - want) <= 1e-10 * np.linalg.norm(want)


def test_newton_schulz_transpose_and_steps():
    rng = np.random.default_rng(9)
    X = rng.standard_normal((30, 50))
    assert np.allclose(M.newton_schulz(X.T), M.newton_schulz(X).T, rtol=1e-12, atol=1e-14)
    assert np.allclose(M.newton_schulz(X, steps=0), X / (np.linalg.norm(X) + 1e-7))


def test_golden_worked_block():
    """The stored worked block (tests/golden/adam8_fp8_block.json) still comes out
    of the oracle bit for bit."""
    import json
    import os

    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "adam8_fp8_block.json")))
    u32 = lambda a: np.asarray(a, np.uint32).view(np.float32)  # noqa: E731
    hp = A.adam_hparams(1e-3, 0.9, 0.999, 1e-8, 10)
    p1, qm1, qv1, sm1, sv1 = A.adam8_block(np.asarray(g["grad_bits"], np.uint16), u32(g["p"]),
                                           np.asarray(g["qm"], np.int8), np.asarray(g["qv"], np.uint8),
                                           np.float32(g["sm"]), np.float32(g["sv"]), hp)
    assert np.array_equal(p1.view(np.uint32), np.asarray(g["out_p"], np.uint32))
    assert qm1.tolist() == g["out_qm"] and qv1.tolist() == g["out_qv"]
    assert int(np.float32(sm1).view(np.uint32)) == g["out_sm"]
    q8, s8 = F.fp8_tile(p1[:128])
    assert q8.tolist() == g["fp8_codes"] and int(np.float32(s8).view(np.uint32)) == g["fp8_scale"]


def test_dequant_view_pins():
    """The bf16 view after the AllGather: exact for power-of-two scales (the
    decoded code times 2^k is exact, then one bf16 rounding of an E4M3 value,
    which bf16 holds exactly); zero scale gives signed zeros; round trip through
    the quantiser within E4M3's half-ulp (2^-4 relative for normals) plus bf16's
    2^-9; only FP8 tiles are written."""
    from oracle import codecs as OC
    from oracle import fp8 as OF

    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]  # the two NaN patterns
    dec = OC.e4m3_decode(codes).astype(np.float32)
    for k in (-20, -3, 0, 5):
        got = OC.bf16_bits_to_f32(OF.dequant_tile(codes, np.float32(2.0 ** k)))
        assert np.array_equal(got, dec * np.float32(2.0 ** k))
    z = OC.bf16_bits_to_f32(OF.dequant_tile(codes, np.float32(0)))
    assert np.all(z == 0) and np.array_equal(np.signbit(z), np.signbit(dec))
    rng = np.random.default_rng(8)
    p = rng.normal(0, 0.02, 128 * 128).astype(np.float32)
    q, s = OF.fp8_tile(p)
    back = OC.bf16_bits_to_f32(OF.dequant_tile(q, s))
    amax = np.abs(p).max()
    normal = np.abs(p) * (448.0 / amax) >= 2.0 ** -6  # scaled value in E4M3's normal range
    rel = np.abs(back[normal] - p[normal]) / np.abs(p[normal])
    assert rel.max() <= 2.0 ** -4 + 2.0 ** -8
    if (~normal).any():  # subnormal codes: half the 2^-9 step, in scaled units
        assert np.abs(back[~normal] - p[~normal]).max() <= 2.0 ** -10 * s * (1 + 2.0 ** -6) + 2.0 ** -9 * np.abs(p[~normal]).max()
    # layout level: FP8 tiles written, everything else untouched
    from oracle import planner as P

    descs = [P.TensorDesc(256, 256, 128 * 256, P.ADAM_FLAT256, True), P.TensorDesc(1, 512, 256, P.ADAM_FLAT256, False)]
    L = P.plan(descs, 2, 128, 16)
    n = 2 * L.S
    master = rng.normal(0, 0.02, n).astype(np.float32)
    qb, sb = OF.quant_fp8(L, 0, 2, master, np.zeros(n, np.uint8), np.zeros(L.n_fslots, np.float32))
    out = OF.dequant_fp8(L, 0, 2, qb, sb, np.full(n, 0x7FC1, np.uint16))
    t0 = L.starts[0]
    assert np.all(out[:t0] == 0x7FC1) and np.all(out[t0 + 256 * 256:] == 0x7FC1)
    err = np.abs(OC.bf16_bits_to_f32(out[t0:t0 + 65536]) - master[t0:t0 + 65536])
    assert err.max() <= 2.0 ** -4 * np.abs(master[t0:t0 + 65536]).max()
