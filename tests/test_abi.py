"""The C ABI on the host (no GPU): the library loads and exports every entry point
include/bq.h declares, the C++ planner's exported table equals the oracle's bit
for bit, and host-detectable errors come back as codes."""

import ctypes as C
import os
import re

import numpy as np
import pytest

import block_quant_gb300 as bq
import workloads as W
from oracle import planner as P

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bq.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_quant_gb300 import build

    build.build()
    return bq.load()


def test_exports_every_declared_symbol(built):
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)  # drop comments
    declared = sorted(set(re.findall(r"\b(bq_[a-z0-9_]+)\s*\(", src)))
    assert declared, "no declarations found"
    assert sorted(bq.SYMBOLS) == declared
    for name in declared:
        assert hasattr(built, name), name
    assert built.bq_version() == 1
    assert built.bq_strerror(bq.BQ_EALIGN) == b"misaligned pointer or offset"


def _oracle_export(descs, V, alpha, start_align):
    return np.asarray(P.plan(descs, V, alpha, start_align).export(), np.int64)


def _descs(unit):
    return [P.TensorDesc(t.rows, t.cols, t.g, t.adam_kind, t.fp8) for t in unit.tensors]


@pytest.mark.parametrize("name", W.NAMED[:4] + W.SMALL[1:4] + W.TILE32 + W.MUON_STEP)
def test_planner_matches_oracle_on_configs(name):
    c = W.config(name)
    for u in c.units:
        want = _oracle_export(_descs(u), c.V, c.alpha, c.start_align)
        got = bq.plan(u.tensors, c.V, c.alpha, c.start_align).export()
        assert np.array_equal(got, want), (name, u.name)


def test_planner_matches_oracle_on_random_groups():
    rng = np.random.default_rng(17)
    for trial in range(300):
        N = int(rng.integers(1, 9))
        descs = []
        for _ in range(N):
            if rng.random() < 0.4:  # 1-D
                rows, cols = 1, int(rng.integers(1, 3000))
                kind = int(rng.integers(0, 2))
                unit = 256 if kind == 0 else 128
                g = unit * int(rng.choice([1, 2, 3]))
                fp8 = bool(rng.random() < 0.5)
            else:
                rows = int(rng.integers(1, 700))
                cols = 8 * int(rng.integers(1, 90))
                kind = int(rng.integers(0, 2))
                band = 128 * cols
                g = band * int(rng.choice([1, 2]))
                if kind == 0:
                    g = int(np.lcm(g, 256))
                fp8 = bool(rng.random() < 0.7)
            descs.append(P.TensorDesc(rows, cols, g, kind, fp8))
        V = int(rng.integers(1, 17))
        alpha = int(rng.choice([1, 8, 128, 1000]))
        align = int(rng.choice([1, 8, 16]))
        want = _oracle_export(descs, V, alpha, align)
        got = bq.plan(descs, V, alpha, align).export()
        assert np.array_equal(got, want), (trial, [(d.rows, d.cols, d.g, d.adam_kind, d.fp8) for d in descs], V)


def test_planner_tiny_granularities_match_oracle():
    rng = np.random.default_rng(23)
    for _ in range(500):
        N = int(rng.integers(1, 7))
        gs = [int(rng.choice([256, 512, 768])) for _ in range(N)]
        ns = [int(rng.integers(1, 9)) * 256 + int(rng.integers(0, 300)) for _ in range(N)]
        descs = [P.TensorDesc(1, n, g, 0, False) for n, g in zip(ns, gs)]
        V = int(rng.integers(1, 8))
        got = bq.plan(descs, V, 1, 1).export()
        assert np.array_equal(got, _oracle_export(descs, V, 1, 1))


def test_planner_rejects_bad_descriptors():
    with pytest.raises(bq.BQError) as e:
        bq.plan([(1, 1000, 100, bq.ADAM_FLAT256, 0)], 4)  # g not a multiple of 256
    assert e.value.code == bq.BQ_EINVAL
    with pytest.raises(bq.BQError) as e:
        bq.plan([(256, 100, 128 * 100, bq.ADAM_TILE128, 1)], 4)  # cols % 8 != 0 for 2-D tiles
    assert e.value.code == bq.BQ_EINVAL
    with pytest.raises(bq.BQError) as e:
        bq.plan([(256, 64, 64, bq.ADAM_TILE128, 0)], 4)  # g splits a 128-row band
    assert e.value.code == bq.BQ_EINVAL
    with pytest.raises(bq.BQError) as e:
        bq.plan([], 4)
    assert e.value.code == bq.BQ_EINVAL
    with pytest.raises(bq.BQError) as e:
        bq.plan([(1, 256, 256, 7, 0)], 4)
    assert e.value.code == bq.BQ_EINVAL


def test_export_needs_room_and_upload_checks_alignment(built):
    L = bq.plan([(1, 1000, 256, 0, 0), (1, 999, 256, 0, 0)], 3, alpha=1, start_align=1)
    buf = np.zeros(5, np.int64)
    rc = built.bq_layout_export(L.handle, buf.ctypes.data_as(C.POINTER(C.c_int64)), 5)
    assert rc == bq.BQ_ENOSPC
    info = L.info()
    # start_align 1 leaves a local offset that is not a multiple of 8: the step
    # kernels refuse such a layout before touching the device
    iv = W.Table(L.export()).intervals
    if np.any(iv[:, 4] % 8):
        with pytest.raises(bq.BQError) as e:
            L.upload_bytes(0, info["V"])
        assert e.value.code == bq.BQ_EALIGN
    with pytest.raises(bq.BQError) as e:
        L.upload_bytes(2, 1)
    assert e.value.code == bq.BQ_EINVAL
    L2 = bq.plan([(1, 1000, 256, 0, 0)], 2)
    assert L2.upload_bytes(0, 2) > 0
    with pytest.raises(bq.BQError) as e:
        L2.upload(0, 2, 0, 1 << 20, stream=0)  # NULL workspace
    assert e.value.code == bq.BQ_EALIGN


def test_layout_info_consistent():
    c = W.config("gptoss-small")
    L = bq.plan(c.units[0].tensors, c.V, c.alpha, c.start_align)
    inf = L.info()
    t = W.Table(L.export())
    assert inf["S"] == t.S and inf["n_intervals"] == t.NI and inf["n_mslots"] == t.n_mslots
    assert inf["total_elems"] == sum(x.numel for x in c.units[0].tensors)
    assert inf["padding_elems"] == c.V * inf["S"] - inf["total_elems"]


def test_shard_tables_pass_host_bounds_check():
    """bq_layout_upload_bytes builds the kernels' work tables and checks every
    element range and scale slot against the shard range on the host; run it on
    every layout the GPU tests use, at every device range they use."""
    import sys

    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from test_parity_step import _edge_tensors

    cases = []
    for name in W.NAMED[:4] + W.SMALL[:4] + W.TILE32 + W.MUON_STEP:
        c = W.config(name)
        for u in c.units:
            cases.append((u.tensors, c.V, c.alpha, c.start_align))
    for V in (1, 2, 3, 5, 6):
        cases.append((_edge_tensors(), V, 128, 16))
    for tensors, V, alpha, align in cases:
        L = bq.plan(tensors, V, alpha, align)
        ranges = {(0, V), (0, 1), (V - 1, V), (V // 2, V)}
        for lo, hi in ranges:
            if lo < hi:
                assert L.upload_bytes(lo, hi) > 0


def test_fastdiv_formula():
    """The kernels divide by a region's column count with a multiply and a shift
    (Granlund-Montgomery): floor(n / d) == (n * m) >> (32 + l - 1) with
    l = ceil(log2 d), m = ceil(2^(31+l) / d), for 0 <= n < 2^31.  Checked here
    for the host-side constants on edge and random cases."""
    rng = np.random.default_rng(3)
    ds = [2, 3, 5, 7, 8, 24, 360, 720, 2880, 4096, 5760, 14336, 28672, (1 << 23) - 1, 1 << 23]
    ds += [int(x) for x in rng.integers(2, 1 << 24, 200)]
    for d in ds:
        l = (d - 1).bit_length()
        m = ((1 << (31 + l)) + d - 1) // d
        assert m < (1 << 32)
        ns = [0, 1, d - 1, d, d + 1, (1 << 31) - 1, (1 << 31) - d] + [int(x) for x in rng.integers(0, 1 << 31, 2000)]
        for n in ns:
            assert ((n * m) >> 32) >> (l - 1) == n // d, (n, d)


def test_muon_roots_and_layout_match_oracle(built):
    """Host logic of the Muon path: the library's root assignment and exported
    layout equal the oracle's on random groups mixing Muon and Adam tensors."""
    import block_quant_gb300 as bq
    from oracle import muon as OM

    rng = np.random.default_rng(11)
    for _ in range(200):
        V = int(rng.integers(1, 7))
        descs = []
        for _ in range(int(rng.integers(1, 12))):
            r, c = (int(x) for x in rng.integers(2, 40, 2) * 8)
            kind = int(rng.choice([0, 2, 2, 3]))
            descs.append((r, c, {0: 256 * c, 2: c, 3: 32 * c}[kind], kind, 0))
        L = bq.plan(descs, V, 128, 16)
        od = [P.TensorDesc(*d[:4]) for d in descs]
        assert list(bq.muon_roots(L)) == OM.muon_roots(od, V)
        assert np.array_equal(L.export(), np.asarray(P.plan(od, V, 128, 16).export(), np.int64))
    with pytest.raises(bq.BQError):
        bq.plan([(1, 256, 256, 2, 0)], 2, 128, 16)  # Muon tensors are 2-D
    with pytest.raises(bq.BQError):
        bq.plan([(256, 256, 256, 2, 1)], 2, 128, 16)  # and take no FP8


def test_placement_orders_match_oracle(built):
    """The three placement orders (given, by block size, by shape) give the
    oracle's layout bit for bit, on the configurations and on random groups."""
    for name in W.NAMED[:4] + W.SMALL[1:4] + W.TILE32:
        c = W.config(name)
        for u in c.units:
            for order in (bq.ORDER_BLOCK, bq.ORDER_SHAPE):
                want = np.asarray(P.plan(_descs(u), c.V, c.alpha, c.start_align, order).export(), np.int64)
                got = bq.plan(u.tensors, c.V, c.alpha, c.start_align, order).export()
                assert np.array_equal(got, want), (name, u.name, order)
    rng = np.random.default_rng(29)
    for _ in range(200):
        descs = []
        for _ in range(int(rng.integers(1, 10))):
            r, cc = int(rng.integers(1, 300)), 8 * int(rng.integers(1, 60))
            g = 256 if r == 1 else int(np.lcm(256, cc * int(rng.choice([1, 8, 128]))))
            descs.append(P.TensorDesc(r, cc, g, 0, False))
        V = int(rng.integers(1, 20))
        for order in (0, 1, 2):
            want = np.asarray(P.plan(descs, V, 128, 16, order).export(), np.int64)
            assert np.array_equal(bq.plan(descs, V, 128, 16, order).export(), want)
    with pytest.raises(bq.BQError):
        bq.plan([(1, 256, 256, 0, 0)], 2, order=3)


def test_adam_hparams_match_oracle(built):
    """The library derives 1-b and the reciprocal bias corrections itself; its
    fp32 values equal the oracle's bit for bit (so a C caller needs no arithmetic
    of its own), and nonsense hyper-parameters come back as BQ_EINVAL."""
    from oracle import adam8 as OA

    for t in (1, 2, 10, 999, 10 ** 6):
        for lr, b1, b2, eps in ((1e-3, 0.9, 0.999, 1e-8), (3e-4, 0.95, 0.98, 1e-6), (0.1, 0.0, 0.5, 0.0)):
            got = bq.adam_hparams(lr, b1, b2, eps, t)
            want = OA.adam_hparams(lr, b1, b2, eps, t)
            for k, v in want.items():
                assert np.float32(getattr(got, k)).tobytes() == v.tobytes(), (k, t, lr)
    hp = bq.AdamHp()
    for args in ((1e-3, 0.9, 0.999, 1e-8, 0), (1e-3, 1.0, 0.999, 1e-8, 1), (1e-3, 0.9, -0.1, 1e-8, 1),
                 (float("nan"), 0.9, 0.999, 1e-8, 1), (1e-3, 0.9, 0.999, float("inf"), 1)):
        assert built.bq_adam_hparams(*args, C.byref(hp)) == bq.BQ_EINVAL, args
    assert built.bq_adam_hparams(1e-3, 0.9, 0.999, 1e-8, 1, None) == bq.BQ_EINVAL


def test_group_place_and_errors(built):
    """Member bases in a group: elements at multiples of 256 in member order
    (each after the previous member's range), slots and tensors back to back;
    a NULL layout, an empty group or a bad range is refused."""
    c = W.config("llama-small")
    lay = bq.plan(c.units[0].tensors, c.V, c.alpha, c.start_align)
    toy = W.config("toy")
    lay2 = bq.plan(toy.units[0].tensors, toy.V, toy.alpha, toy.start_align)
    T, T2 = W.Table(lay.export()), W.Table(lay2.export())
    members = [(lay, 0, 8), (lay2, 1, 3), (lay, 3, 5)]
    g = bq.Group(members)
    end = ms = fs = nt = 0
    for (L, lo, hi), tab, p in zip(members, (T, T2, T), g.place):
        eb = -(-end // 256) * 256
        assert p == dict(elem_base=eb, mslot_base=ms, fslot_base=fs, tensor_base=nt)
        end = eb + (hi - lo) * tab.S
        a, b = tab.slot_range(lo, hi)
        ms += b - a
        a, b = tab.slot_range(lo, hi, fp8=True)
        fs += b - a
        nt += tab.N
    assert g.info == dict(elems=end, mslots=ms, fslots=fs, tensors=nt)
    assert g.upload_bytes() > 0
    bad = (bq.Member * 1)(bq.Member(None, 0, 1))
    assert built.bq_group_place(bad, 1, None, None) == bq.BQ_EINVAL
    assert built.bq_group_place(bad, 0, None, None) == bq.BQ_EINVAL
    bad = (bq.Member * 1)(bq.Member(lay.handle.value, 5, 9))
    assert built.bq_group_place(bad, 1, None, None) == bq.BQ_EINVAL
    n = C.c_size_t()
    assert built.bq_group_upload_bytes(bad, 1, C.byref(n)) == bq.BQ_EINVAL
