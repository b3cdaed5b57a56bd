"""The two exchanges around the DBuffer step, over torch.distributed.

RaggedShard makes every local shard of a DBuffer the same size S and contiguous
(veScale-FSDP, feynmanwiki walkthrough, paper section 5, DBuffer paragraphs:
the collectives run on the buffer in place, with no copy-in before or copy-out
after them).  So the exchanges of a data-parallel step are single calls on
slices of caller buffers:

  * before the optimizer step, ReduceScatter of the packed bf16 gradient
    DBuffer: every rank holds the whole buffer (V*S elements, bq_pack over all
    V devices) and receives the sum over ranks of its own devices' slice;
  * after it, AllGather of the FP8 staging buffer (each rank's slice, the same
    length on every rank) and of the FP8 tile scales (a ragged number of slots
    per rank: exchanged padded to the longest rank, then trimmed).

Ranks own equal runs of consecutive devices: rank r of W owns devices
[r*V/W, (r+1)*V/W) (V % W == 0).

The n-D DBuffer (same passage: a DBuffer sharded over one mesh dimension and
replicated over another) adds one exchange: on a mesh of R replicas x W shards
(rank = replica * W + shard), the ReduceScatter runs inside each replica's shard
group and an AllReduce of the reduced slice runs across the replicas holding the
same shard; the AllGather stays inside the shard group.

Nothing here computes any of the method's arithmetic: the reduction is the
collective's sum, everything else moves bytes.  The calls are torch.distributed
collectives on the caller's tensors (NCCL on GPUs; tested on CPU ranks over
gloo).
"""

import numpy as np


def rank_devices(V, world, rank):
    """Devices [dev_lo, dev_hi) owned by `rank` of `world` ranks."""
    if world < 1 or V % world or not 0 <= rank < world:
        raise ValueError(f"need V % world == 0 and 0 <= rank < world (V={V}, world={world}, rank={rank})")
    k = V // world
    return rank * k, (rank + 1) * k


def mesh_groups(replicas, shards):
    """The process groups of a replicas x shards mesh (rank = replica * shards +
    shard): this rank's shard group (the ranks of its replica) and replica group
    (the ranks holding its shard), created collectively on every rank."""
    import torch.distributed as dist

    rank = dist.get_rank()
    if dist.get_world_size() != replicas * shards:
        raise ValueError("the world is not replicas x shards")
    shard_group = replica_group = None
    for r in range(replicas):  # every rank creates every group, in the same order
        g = dist.new_group([r * shards + s for s in range(shards)])
        if rank // shards == r:
            shard_group = g
    for s in range(shards):
        g = dist.new_group([r * shards + s for r in range(replicas)])
        if rank % shards == s:
            replica_group = g
    return shard_group, replica_group


def reduce_scatter_allreduce_grad(full, local, shard_group, replica_group):
    """n-D DBuffer: local <- this rank's slice summed over its shard group, then
    summed over its replica group (in place)."""
    import torch.distributed as dist

    reduce_scatter_grad(full, local, group=shard_group)
    dist.all_reduce(local, op=dist.ReduceOp.SUM, group=replica_group)


def device_table(layout):
    """Per device k of the layout (and k = V): [first interval, first Adam slot,
    first FP8 slot], read from the layout's exported table (int64, (V+1) x 3)."""
    ex = layout.export()
    V, N, NI = int(ex[2]), int(ex[4]), int(ex[5])
    o = 8 + 7 * N + 7 * NI
    return ex[o:o + 3 * (V + 1)].reshape(V + 1, 3)


def reduce_scatter_grad(full, local, group=None):
    """local <- this rank's devices' slice of the sum over ranks of `full`.
    full: the packed gradient DBuffer of all V devices; local: (V/W)*S
    elements of the same dtype."""
    import torch.distributed as dist

    if full.numel() != local.numel() * dist.get_world_size(group):
        raise ValueError("full must hold world_size equal slices of local's size")
    dist.reduce_scatter_tensor(local, full, op=dist.ReduceOp.SUM, group=group)


def all_gather_fp8(local, full, group=None):
    """full <- every rank's FP8 staging slice in rank order (device order)."""
    import torch.distributed as dist

    if full.numel() != local.numel() * dist.get_world_size(group):
        raise ValueError("full must hold world_size slices of local's size")
    dist.all_gather_into_tensor(full, local, group=group)


def all_gather_scales(layout, local, full, fp8=True, group=None):
    """full <- the scale slots of every device (FP8 tile scales, or Adam block
    scales with fp8=False).  local holds this rank's slots (slot z of its first
    device at index 0); ranks hold different numbers of slots, so the slices
    travel padded to the longest one and are trimmed on arrival."""
    import torch
    import torch.distributed as dist

    world, rank = dist.get_world_size(group), dist.get_rank(group)
    dt = device_table(layout)
    V = dt.shape[0] - 1
    col = 2 if fp8 else 1
    bounds = [rank_devices(V, world, r) for r in range(world)]
    counts = [int(dt[hi, col] - dt[lo, col]) for lo, hi in bounds]
    if local.numel() < counts[rank] or full.numel() < int(dt[V, col]):
        raise ValueError("scale buffers too small for the layout's slots")
    width = max(max(counts), 1)
    send = torch.zeros(width, dtype=local.dtype, device=local.device)
    send[:counts[rank]] = local[:counts[rank]]
    recv = torch.empty(width * world, dtype=local.dtype, device=local.device)
    dist.all_gather_into_tensor(recv, send, group=group)
    for r, (lo, hi) in enumerate(bounds):
        z0 = int(dt[lo, col])
        full[z0:z0 + counts[r]] = recv[r * width:r * width + counts[r]]
    return np.asarray(counts)
