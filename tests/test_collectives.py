"""The exchanges around the DBuffer step on CPU ranks over gloo (world_size 2, and
a 2 x 2 replicas x shards mesh for the n-D DBuffer).

Each rank packs its own gradients into the whole DBuffer (all V devices), the
ReduceScatter gives it the summed slice of its own devices, it runs the step
(the oracle stands in for the kernels, which need a GPU) on those devices only,
and the AllGathers assemble the FP8 staging buffer and the scale slots.  The
result must equal, bit for bit, one process running the oracle over all V
devices on the summed gradients: the partitioning of devices over ranks, the
in-place slices and the ragged scale exchange lose nothing."""

import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(name, rank_of_grads):
    """The configuration, both layouts and one rank's whole-tensor gradients."""
    import workloads as W
    from oracle import planner as P

    import block_quant_gb300 as bq

    c = W.config(name)
    unit = c.units[0]
    olay = P.plan([P.TensorDesc(t.rows, t.cols, t.g, t.adam_kind, t.fp8) for t in unit.tensors], c.V, c.alpha,
                  c.start_align)
    lay = bq.plan(unit.tensors, c.V, c.alpha, c.start_align)
    assert np.array_equal(lay.export(), np.asarray(olay.export(), np.int64))
    grads = {i: (W.grad_bits(c.cfg_id + 100 * (rank_of_grads + 1), 0, i, 0, t.numel), 0)
             for i, t in enumerate(unit.tensors) if t.numel}
    return c, olay, lay, grads


def _state(c, T, lo, hi):
    import workloads as W

    cid = c.cfg_id
    master = W.scatter_local(T, lo, hi, lambda i, a, b: W.master_values(cid, 0, i, a, b), np.float32)
    m = W.scatter_local(T, lo, hi, lambda i, a, b: W.mcode_values(cid, 0, i, a, b), np.int8)
    v = W.scatter_local(T, lo, hi, lambda i, a, b: W.vcode_values(cid, 0, i, a, b), np.uint8)
    m0, m1 = T.slot_range(lo, hi)
    return master, m, v, W.scale_values(cid, 0, "m", m0, m1), W.scale_values(cid, 0, "v", m0, m1)


def _step(c, olay, T, lo, hi, dbuf):
    """The oracle's Adam + FP8 over devices [lo, hi) from a packed gradient slice."""
    from oracle import adam8 as OA
    from oracle import fp8 as OF

    master, m, v, ms, vs = _state(c, T, lo, hi)
    hp = OA.adam_hparams(c.lr, c.b1, c.b2, c.eps, c.t)
    master, m, v, ms, vs = OA.adam8_step(olay, lo, hi, dbuf, master, m, v, ms, vs, hp)
    f0, f1 = T.slot_range(lo, hi, fp8=True)
    q, fs = OF.quant_fp8(olay, lo, hi, master, np.zeros((hi - lo) * T.S, np.uint8), np.zeros(f1 - f0, np.float32))
    return q, fs, ms, vs


def _worker(rank, world, port, name, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import workloads as W
    from block_quant_gb300 import collectives as X
    from oracle import pack as OP

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c, olay, lay, grads = _inputs(name, rank)
        T = W.Table(lay.export())
        V, S = c.V, T.S
        lo, hi = X.rank_devices(V, world, rank)
        sc = np.float32(1.0 / world)
        # the whole DBuffer of this rank's gradients, packed (all V devices)
        full = OP.pack(olay, 0, V, grads, np.zeros(V * S, np.uint16), sc, False)
        t_full = torch.from_numpy(full.view(np.int16)).view(torch.bfloat16)
        t_local = torch.empty((hi - lo) * S, dtype=torch.bfloat16)
        X.reduce_scatter_grad(t_full, t_local)
        local = t_local.view(torch.int16).numpy().view(np.uint16)
        # this rank's step on its own devices, then the AllGathers
        q8, fs, ms, vs = _step(c, olay, T, lo, hi, local)
        t_q = torch.empty(V * S, dtype=torch.uint8)
        X.all_gather_fp8(torch.from_numpy(q8), t_q)
        nf, nm = T.slot_range(0, V, fp8=True)[1], T.slot_range(0, V)[1]
        g_fs, g_ms, g_vs = torch.zeros(nf), torch.zeros(nm), torch.zeros(nm)
        X.all_gather_scales(lay, torch.from_numpy(fs), g_fs, fp8=True)
        X.all_gather_scales(lay, torch.from_numpy(ms), g_ms, fp8=False)
        X.all_gather_scales(lay, torch.from_numpy(vs), g_vs, fp8=False)
        q.put((rank, local, t_q.numpy(), g_fs.numpy(), g_ms.numpy(), g_vs.numpy(), None))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, None, None, None, None, None, repr(e)))
    finally:
        dist.destroy_process_group()


def _run(name, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, name, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        r = q.get(timeout=600)
        out[r[0]] = r[1:]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r, res in out.items():
        assert res[-1] is None, f"rank {r}: {res[-1]}"
    return out


def test_reduce_scatter_and_all_gather_equal_the_v_shard_oracle():
    sys.path.insert(0, ROOT)
    import workloads as W
    from block_quant_gb300 import collectives as X
    from oracle import codecs as OC
    from oracle import pack as OP

    name, world = "llama-small", 2
    out = _run(name, world)
    # expected: one process, the summed gradient of both ranks over all V devices
    c, olay, lay, g0 = _inputs(name, 0)
    _, _, _, g1 = _inputs(name, 1)
    T = W.Table(lay.export())
    V, S = c.V, T.S
    sc = np.float32(1.0 / world)
    p0 = OP.pack(olay, 0, V, g0, np.zeros(V * S, np.uint16), sc, False)
    p1 = OP.pack(olay, 0, V, g1, np.zeros(V * S, np.uint16), sc, False)
    summed = OC.f32_to_bf16_bits(OC.bf16_bits_to_f32(p0) + OC.bf16_bits_to_f32(p1))  # one rounded add
    for r in range(world):
        lo, hi = X.rank_devices(V, world, r)
        assert np.array_equal(out[r][0], summed[lo * S:hi * S]), f"rank {r}: ReduceScatter slice"
    q8, fs, ms, vs = _step(c, olay, T, 0, V, summed)
    for r in range(world):
        _, g_q, g_fs, g_ms, g_vs, _ = out[r]
        assert np.array_equal(g_q, q8), f"rank {r}: gathered FP8 codes"
        assert np.array_equal(g_fs.view(np.uint32), fs.view(np.uint32)), f"rank {r}: gathered FP8 scales"
        assert np.array_equal(g_ms.view(np.uint32), ms.view(np.uint32)), f"rank {r}: gathered m scales"
        assert np.array_equal(g_vs.view(np.uint32), vs.view(np.uint32)), f"rank {r}: gathered v scales"


def test_rank_devices_and_device_table():
    sys.path.insert(0, ROOT)
    import pytest

    import workloads as W
    from block_quant_gb300 import collectives as X

    import block_quant_gb300 as bq

    assert X.rank_devices(8, 2, 1) == (4, 8) and X.rank_devices(64, 64, 5) == (5, 6)
    with pytest.raises(ValueError):
        X.rank_devices(6, 4, 0)
    c = W.config("gptoss-small")
    lay = bq.plan(c.units[0].tensors, c.V, c.alpha, c.start_align)
    T = W.Table(lay.export())
    assert np.array_equal(X.device_table(lay), T.devices)


def _mesh_worker(rank, world, port, name, replicas, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import workloads as W
    from block_quant_gb300 import collectives as X
    from oracle import pack as OP

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shards = world // replicas
        sg, rg = X.mesh_groups(replicas, shards)
        c, olay, lay, grads = _inputs(name, rank)
        T = W.Table(lay.export())
        V, S = c.V, T.S
        lo, hi = X.rank_devices(V, shards, rank % shards)
        full = OP.pack(olay, 0, V, grads, np.zeros(V * S, np.uint16), np.float32(1.0 / world), False)
        t_local = torch.empty((hi - lo) * S, dtype=torch.bfloat16)
        X.reduce_scatter_allreduce_grad(torch.from_numpy(full.view(np.int16)).view(torch.bfloat16), t_local, sg, rg)
        local = t_local.view(torch.int16).numpy().view(np.uint16)
        q8, fs, ms, vs = _step(c, olay, T, lo, hi, local)
        t_q = torch.empty(V * S, dtype=torch.uint8)
        X.all_gather_fp8(torch.from_numpy(q8), t_q, group=sg)
        g_fs = torch.zeros(T.slot_range(0, V, fp8=True)[1])
        X.all_gather_scales(lay, torch.from_numpy(fs), g_fs, fp8=True, group=sg)
        q.put((rank, local, t_q.numpy(), g_fs.numpy(), None))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, None, None, None, repr(e)))
    finally:
        dist.destroy_process_group()


def test_n_d_dbuffer_mesh_equals_the_v_shard_oracle():
    """A 2 x 2 mesh (2 replicas x 2 shards): ReduceScatter inside the shard group,
    AllReduce across the replicas, the step on the rank's devices, AllGather inside
    the shard group.  Every rank ends with the FP8 buffer and scales of one process
    running the oracle over all V devices on the same two-level sum."""
    sys.path.insert(0, ROOT)
    import workloads as W
    from block_quant_gb300 import collectives as X
    from oracle import codecs as OC
    from oracle import pack as OP

    name, world, replicas = "gptoss-small", 4, 2
    shards = world // replicas
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_mesh_worker, args=(r, world, port, name, replicas, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        r = q.get(timeout=600)
        out[r[0]] = r[1:]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r, res in out.items():
        assert res[-1] is None, f"rank {r}: {res[-1]}"
    c, olay, lay, _ = _inputs(name, 0)
    T = W.Table(lay.export())
    V, S = c.V, T.S
    sc = np.float32(1.0 / world)
    packed = [OP.pack(olay, 0, V, _inputs(name, r)[3], np.zeros(V * S, np.uint16), sc, False) for r in range(world)]
    f = OC.bf16_bits_to_f32
    # the sum inside each replica's shard group, then across the replicas (each a single rounded add)
    per_replica = [OC.f32_to_bf16_bits(f(packed[rr * shards]) + f(packed[rr * shards + 1])) for rr in range(replicas)]
    summed = OC.f32_to_bf16_bits(f(per_replica[0]) + f(per_replica[1]))
    for r in range(world):
        lo, hi = X.rank_devices(V, shards, r % shards)
        assert np.array_equal(out[r][0], summed[lo * S:hi * S]), f"rank {r}: reduced slice"
    q8, fs, _, _ = _step(c, olay, T, 0, V, summed)
    for r in range(world):
        assert np.array_equal(out[r][1], q8), f"rank {r}: gathered FP8 codes"
        assert np.array_equal(out[r][2].view(np.uint32), fs.view(np.uint32)), f"rank {r}: gathered FP8 scales"
