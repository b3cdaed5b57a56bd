"""Pins of the oracle's Muon step around Newton-Schulz (no GPU): root assignment
against a brute-force optimum (Graham's bound for longest-first greedy), the
Newton-Schulz cost against the product shapes, momentum and apply against exact
rational arithmetic and closed forms, the gather against the packed gradients,
and the planner's treatment of Muon tensors (no Adam blocks, slots or FP8)."""

import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import codecs as OC
from oracle import muon as OM
from oracle import pack as OP
from oracle import planner as P


def _random_muon_descs(rng, n):
    out = []
    for _ in range(n):
        r, c = (int(x) for x in rng.integers(2, 9, 2) * 16)
        out.append(P.TensorDesc(r, c, c, P.OPT_MUON))
    return out


def test_ns_cost_counts_the_three_products():
    """One step: A = X X^T (m x n by n x m), A A (m^3), B X (m x m by m x n), each
    2 M N K flops, with X the wide orientation (m = min dim)."""
    for rows, cols in [(4096, 4096), (4096, 14336), (14336, 4096), (3, 7), (1024, 8192)]:
        m, n = min(rows, cols), max(rows, cols)
        products = [(m, m, n), (m, m, m), (m, n, m)]  # (M, N, K)
        assert OM.ns_cost(rows, cols) == sum(2 * a * b * k for a, b, k in products)


def test_roots_within_graham_bound_of_optimum():
    """Longest-first greedy makespan <= (4/3 - 1/(3V)) x optimum (Graham 1969);
    the optimum by exhaustive assignment on tiny instances."""
    rng = np.random.default_rng(3)
    worst = 0.0
    for _ in range(60):
        V = int(rng.integers(2, 4))
        descs = _random_muon_descs(rng, int(rng.integers(2, 7)))
        costs = [OM.ns_cost(d.rows, d.cols) for d in descs]
        roots = OM.muon_roots(descs, V)
        load = [0] * V
        for i, k in enumerate(roots):
            load[k] += costs[i]
        opt = min(max(sum(c for c, k in zip(costs, assign) if k == j) for j in range(V))
                  for assign in itertools.product(range(V), repeat=len(costs)))
        assert max(load) <= (Fraction(4, 3) - Fraction(1, 3 * V)) * opt
        worst = max(worst, max(load) / opt)
    assert worst >= 1.0


def test_roots_cover_muon_tensors_only():
    descs = [P.TensorDesc(1, 256, 256), P.TensorDesc(64, 64, 64, P.OPT_MUON), P.TensorDesc(32, 256, 256),
             P.TensorDesc(128, 64, 64, P.OPT_MUON), P.TensorDesc(64, 64, 64, P.OPT_MUON)]
    roots = OM.muon_roots(descs, 2)
    assert roots[0] == -1 and roots[2] == -1
    # the 128 x 64 matrix is the largest: device 0; the two equal ones then fill
    # device 1 first (least loaded), then device 1 again (its load is still lower)
    assert roots[3] == 0 and roots[1] == 1 and roots[4] == 1
    assert OM.muon_roots(descs, 1) == [-1, 0, -1, 0, 0]
    # equal costs spread round robin
    same = [P.TensorDesc(64, 64, 64, P.OPT_MUON) for _ in range(6)]
    assert OM.muon_roots(same, 3) == [0, 1, 2, 0, 1, 2]


def test_planner_gives_muon_tensors_no_blocks_or_slots():
    descs = [P.TensorDesc(256, 256, 128 * 256, P.OPT_MUON), P.TensorDesc(1, 512, 256),
             P.TensorDesc(256, 512, 128 * 512, P.ADAM_FLAT256, True)]
    L = P.plan(descs, 3, 128, 16)
    assert L.n_mslots == 2 + 512  # the 1-D tensor's 2 blocks + the 2-D Adam tensor's 512
    muon_pos = np.zeros(3 * L.S, bool)
    muon_pos[L.starts[0]:L.starts[0] + descs[0].numel] = True
    for _, pos in P.adam_blocks(L, 0, 3):
        assert not muon_pos[pos].any()
    for _, pos in P.fp8_tiles(L, 0, 3):
        assert not muon_pos[pos].any()
    for p in np.nonzero(muon_pos)[0][::997]:
        assert P.block_at(L, 0, 3, int(p)) is None
    with pytest.raises(ValueError):
        P.plan([P.TensorDesc(256, 256, 256, P.OPT_MUON, True)], 2, 128, 16)
    with pytest.raises(ValueError):
        P.plan([P.TensorDesc(1, 256, 256, P.OPT_MUON)], 2, 128, 16)


def _exact_fma(a, b, c):
    """a*b + c exactly, rounded once to fp32 (Fraction arithmetic)."""
    x = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
    return np.float32(float(x)) if abs(x) < 2 ** 120 else None


def _layout_with_muon():
    descs = [P.TensorDesc(96, 64, 64, P.OPT_MUON), P.TensorDesc(1, 256, 256),
             P.TensorDesc(160, 48, 48, P.OPT_MUON), P.TensorDesc(64, 256, 256)]
    return descs, P.plan(descs, 4, 128, 16)


def _grads(descs, rng):
    return {i: (OC.f32_to_bf16_bits(rng.normal(0, 1e-2, d.numel).astype(np.float32)), 0)
            for i, d in enumerate(descs)}


def test_momentum_closed_forms():
    descs, L = _layout_with_muon()
    n = L.V * L.S
    one = {i: (np.full(d.numel, 0x3F80, np.uint16), 0) for i, d in enumerate(descs)}  # bf16 1.0
    dbuf = OP.pack(L, 0, L.V, one, np.zeros(n, np.uint16), np.float32(1.0), False)
    mom = np.zeros(n, np.float32)
    for t in range(1, 12):
        mom, _ = OM.muon_momentum(L, 0, L.V, dbuf, mom, 0.5)
        want = np.float32(2.0 - 2.0 ** (1 - t))  # 1 + 1/2 + ... + 2^(1-t)
        for pos, i, t_off, ln in OM._muon_pieces(L, 0, L.V):
            assert np.all(mom[pos:pos + ln] == want)
    # mu = 0: M = G exactly, whatever M held
    rng = np.random.default_rng(1)
    dbuf = OP.pack(L, 0, L.V, _grads(descs, rng), np.zeros(n, np.uint16), np.float32(1.0), False)
    m1, _ = OM.muon_momentum(L, 0, L.V, dbuf, rng.normal(0, 1, n).astype(np.float32), 0.0)
    for pos, i, t_off, ln in OM._muon_pieces(L, 0, L.V):
        assert np.array_equal(m1[pos:pos + ln], OC.bf16_bits_to_f32(dbuf[pos:pos + ln]))


def test_momentum_exact_and_non_muon_untouched():
    descs, L = _layout_with_muon()
    n = L.V * L.S
    rng = np.random.default_rng(2)
    dbuf = OP.pack(L, 0, L.V, _grads(descs, rng), np.zeros(n, np.uint16), np.float32(1.0), False)
    mom0 = rng.normal(0, 1e-2, n).astype(np.float32)
    mu = 0.95
    mom1, _ = OM.muon_momentum(L, 0, L.V, dbuf, mom0, mu)
    muon = np.zeros(n, bool)
    for pos, i, t_off, ln in OM._muon_pieces(L, 0, L.V):
        muon[pos:pos + ln] = True
    assert np.array_equal(mom1[~muon], mom0[~muon])
    g = OC.bf16_bits_to_f32(dbuf)
    for p in rng.choice(np.nonzero(muon)[0], 400, replace=False):
        assert mom1[p] == _exact_fma(np.float32(mu), mom0[p], g[p])


def test_gather_assembles_each_matrix_in_row_major_order():
    """With mu = 0 and zero momentum, the gathered matrices are the original
    gradients (packed with scale 1): every element once, in row-major order."""
    descs, L = _layout_with_muon()
    n = L.V * L.S
    rng = np.random.default_rng(4)
    grads = _grads(descs, rng)
    dbuf = OP.pack(L, 0, L.V, grads, np.zeros(n, np.uint16), np.float32(1.0), False)
    # gather across two shard ranges, as two roots' inputs would be
    _, ga = OM.muon_momentum(L, 0, 2, dbuf[:2 * L.S], np.zeros(2 * L.S, np.float32), 0.0)
    _, gb = OM.muon_momentum(L, 2, 4, dbuf[2 * L.S:], np.zeros(2 * L.S, np.float32), 0.0)
    for i, d in enumerate(descs):
        if d.adam_kind != P.OPT_MUON:
            assert i not in ga and i not in gb
            continue
        full = OM.assemble(d, ga.get(i, []) + gb.get(i, []))
        assert np.array_equal(full.reshape(-1), grads[i][0])


def test_apply_exact_and_closed_forms():
    descs, L = _layout_with_muon()
    n = L.V * L.S
    rng = np.random.default_rng(5)
    w = rng.normal(0, 0.02, n).astype(np.float32)
    ups = {i: OC.f32_to_bf16_bits(rng.normal(0, 0.05, d.numel).astype(np.float32))
           for i, d in enumerate(descs) if d.adam_kind == P.OPT_MUON}
    lrs = {i: 0.02 for i in ups}
    w1 = OM.muon_apply(L, 0, L.V, w, ups, lrs)
    muon = np.zeros(n, bool)
    for pos, i, t_off, ln in OM._muon_pieces(L, 0, L.V):
        muon[pos:pos + ln] = True
        o = OC.bf16_bits_to_f32(ups[i][t_off:t_off + ln])
        for j in rng.integers(0, ln, 60):
            assert w1[pos + j] == _exact_fma(-np.float32(0.02), o[j], w[pos + j])
    assert np.array_equal(w1[~muon], w[~muon])
    # lr = 0 and O = 0 leave W unchanged
    assert np.array_equal(OM.muon_apply(L, 0, L.V, w, ups, {i: 0.0 for i in ups}), w)
    zeros = {i: np.zeros_like(u) for i, u in ups.items()}
    assert np.array_equal(OM.muon_apply(L, 0, L.V, w, zeros, lrs), w)
