"""RaggedShard layout planner (oracle; test infrastructure only).

The problem, as the feynmanwiki walkthrough of veScale-FSDP states it (paper
section 5, the planning problem and its constraints): tensors of one
communication group, spanning V devices, are laid out in ONE global buffer of size
V*S; every device owns the equal local piece [k*S, (k+1)*S); tensor i occupies one
contiguous interval [s_i, s_i + n_i); intervals do not overlap and padding may only
sit between tensors; whenever a device boundary b = k*S falls strictly inside
tensor i, its offset b - s_i is a multiple of the tensor's atomic block size g_i.
The objective is the smallest S.

The pages' heuristic (Key claims / Method on the bud-325 summary; planner
paragraphs of the walkthrough, paper section 5 Algorithm 1):
  * tensors keep the default order (sorted orders are mentioned, default is used);
  * for a candidate S a dynamic program decides feasibility (f(i, j) = fewest local
    shards holding every tensor before i and the first j blocks of i, feasible if
    it stays within V) and f is monotone in j, so runs of j are skipped;
  * candidate S lie on multiples of an alignment L that starts at the collective
    alignment and absorbs, by least common multiple, the granularity of every
    tensor that fully contains a local shard ("Case 3");
  * the Case-3 sets tried are prefixes of the tensors sorted by element count, and
    S is binary-searched over multiples of L, giving a 2-approximation.

Readings taken where the pages are silent (formulas stripped from the page):
  * feasibility for a fixed order and S is computed as exact earliest-fit: each
    tensor starts at the smallest admissible offset at or after the previous end.
    Because padding may be added anywhere between tensors, an earlier end never
    hurts the tensors that follow, so earliest-fit decides exactly whether the
    DP's final shard count stays within V;
  * the last atomic block of a tensor may be partial; cuts are at multiples of g
    from the tensor start;
  * the binary search's lower bracket is ceil(sum n / V) rounded up to L; the upper
    bracket is found by doubling, capped at sum n + N*start_align rounded up to L
    (always feasible: everything fits on device 0); the answer is the smallest
    multiple found by bisection, assuming monotonicity as the pages do;
  * ties between prefixes go to the shortest prefix;
  * ``start_align`` (a minimum alignment of every tensor start, for vector access)
    is not on the pages; with start_align = 1 it has no effect.
"""

import itertools
import math
from functools import lru_cache

import numpy as np

# Adam block geometry kinds and the flat export format (kept identical, by
# definition, to the library's own; see the export docstring).
ADAM_FLAT256 = 0
ADAM_TILE128 = 1
# 32x32 tiles of the 2-D view (1-D tensors: 32-element blocks): the 8-bit Adam
# blocks of the pages' own experiment (paper section 6.3), with 32-row granularity
ADAM_TILE32 = 3
# a 2-D tensor updated by Muon (momentum, Newton-Schulz at a root, apply): no
# Adam blocks or scale slots, no FP8 staging
OPT_MUON = 2
EXPORT_MAGIC = 0x4251
EXPORT_VERSION = 1


def roundup(x, a):
    return -(-x // a) * a


# ----------------------------------------------------------------------------- feasibility


def earliest_start(e, n, g, S, V, start_align):
    """Smallest admissible start s >= e (s a multiple of start_align) for a tensor
    of n elements and atomic block g in a buffer of V local shards of size S, or
    None if the tensor cannot end within V*S.

    Scan: let b be the first device boundary strictly after s.
      * b >= s + n: no boundary inside the tensor -> admissible.
      * (b - s) mod g = r != 0: no start in [s, s + r) can be admissible (b stays
        inside and its offset is not a block multiple) -> move to s + r.
      * b is aligned but a second boundary b + S is also inside and S mod g != 0:
        the two offsets cannot both be multiples of g for any start before b ->
        move to b.
      * otherwise every interior boundary b + jS sits at a multiple of g.
    """
    total = V * S
    s = roundup(e, start_align)
    while True:
        if s + n > total:
            return None
        b = (s // S + 1) * S
        if b >= s + n:
            return s
        r = (b - s) % g
        if r != 0:
            s = roundup(s + r, start_align)
            continue
        if b + S < s + n and S % g != 0:
            s = roundup(b, start_align)
            continue
        return s


def place(ns, gs, order, S, V, start_align):
    """Earliest-fit placement of the tensors in ``order``; returns the list of
    starts indexed by tensor, or None when S is infeasible for this order."""
    starts = [None] * len(ns)
    e = 0
    for i in order:
        s = earliest_start(e, ns[i], gs[i], S, V, start_align)
        if s is None:
            return None
        starts[i] = s
        e = s + ns[i]
    return starts


# ----------------------------------------------------------------------------- heuristic


def plan_sizes(ns, gs, V, alpha, start_align=1, order=None):
    """The prefix / binary-search heuristic over a fixed placement order (default:
    the given one).  Returns (S, starts, k_best) where k_best is the length of the
    winning Case-3 prefix."""
    N = len(ns)
    if N == 0 or V < 1 or alpha < 1 or start_align < 1:
        raise ValueError("empty group or bad V / alignment")
    if any(n < 0 for n in ns) or any(g < 1 for g in gs):
        raise ValueError("bad tensor size or granularity")
    order = list(range(N)) if order is None else list(order)
    total = sum(ns)
    base_cap = roundup(total + N * start_align, alpha)
    by_size = sorted(range(N), key=lambda i: (-ns[i], i))

    def feasible(S):
        return place(ns, gs, order, S, V, start_align) is not None

    best_S, best_k = None, None
    L = alpha
    for k in range(N + 1):
        if k > 0:
            L = L // math.gcd(L, gs[by_size[k - 1]]) * gs[by_size[k - 1]]
        if L > base_cap:
            break  # every later prefix has an even larger L: none can win
        lb = max(roundup(-(-total // V), L), L)
        cap = roundup(base_cap, L)
        hi = lb
        while hi < cap and not feasible(hi):
            hi = min(hi * 2, cap)
        lo_j, hi_j = lb // L, hi // L
        while lo_j < hi_j:
            mid = (lo_j + hi_j) // 2
            if feasible(mid * L):
                hi_j = mid
            else:
                lo_j = mid + 1
        S_k = hi_j * L
        if best_S is None or S_k < best_S:
            best_S, best_k = S_k, k
    starts = place(ns, gs, order, best_S, V, start_align)
    assert starts is not None
    return best_S, starts, best_k


def linear_scan_min(ns, gs, V, alpha, start_align=1):
    """Smallest multiple of alpha at which the default order is feasible, by
    scanning upward (shows any gap left by the bisection's monotonicity
    assumption)."""
    total = sum(ns)
    S = max(roundup(-(-total // V), alpha), alpha)
    while place(ns, gs, list(range(len(ns))), S, V, start_align) is None:
        S += alpha
    return S


# ----------------------------------------------------------------------------- brute force (pins)


def exists_placement(ns, gs, order, S, V, start_align=1):
    """Exhaustive search: is there ANY start assignment (tensors in ``order``, non
    overlapping, every start a multiple of start_align) meeting the block rule?
    Independent of earliest_start; polynomial thanks to memoisation on
    (position in order, previous end)."""
    total = V * S
    bounds = list(range(S, total, S))

    def ok(s, n, g):
        return all((b - s) % g == 0 for b in bounds if s < b < s + n)

    @lru_cache(maxsize=None)
    def rec(idx, e):
        if idx == len(order):
            return True
        i = order[idx]
        n, g = ns[i], gs[i]
        for s in range(roundup(e, start_align), total - n + 1, start_align):
            if ok(s, n, g) and rec(idx + 1, s + n):
                return True
        return False

    return rec(0, 0)


def brute_force_opt(ns, gs, V, alpha, start_align=1):
    """True optimum over every tensor order and every S (multiple of alpha)."""
    total = sum(ns)
    S = max(roundup(-(-total // V), alpha), alpha)
    perms = list(itertools.permutations(range(len(ns))))
    while True:
        if any(exists_placement(ns, gs, p, S, V, start_align) for p in perms):
            return S
        S += alpha


# ----------------------------------------------------------------------------- invariants


def check_layout(ns, gs, starts, S, V):
    """Raise AssertionError unless the placement meets every constraint of the
    problem statement: inside [0, V*S), non-overlapping, and every device boundary
    inside a tensor at a multiple of its g from the tensor start."""
    total = V * S
    spans = sorted((starts[i], starts[i] + ns[i], i) for i in range(len(ns)))
    prev_end = 0
    for s, e, i in spans:
        assert 0 <= s and e <= total, f"tensor {i} outside the buffer"
        assert s >= prev_end, f"tensor {i} overlaps its predecessor"
        prev_end = e
        for b in range(S, total, S):
            if s < b < e:
                assert (b - s) % gs[i] == 0, f"boundary {b} splits a block of tensor {i}"


# ----------------------------------------------------------------------------- descriptor level


class TensorDesc:
    """rows x cols row-major 2-D view (1-D tensors: rows = 1), atomic block g in
    elements, Adam block geometry and whether the tensor has FP8 tiles."""

    __slots__ = ("rows", "cols", "g", "adam_kind", "fp8")

    def __init__(self, rows, cols, g, adam_kind=ADAM_FLAT256, fp8=False):
        self.rows, self.cols, self.g = int(rows), int(cols), int(g)
        self.adam_kind, self.fp8 = int(adam_kind), bool(fp8)

    @property
    def numel(self):
        return self.rows * self.cols

    def tile_unit(self):
        """Elements per 128-row band of the 2-D view (1-D: one 1x128 tile)."""
        return 128 if self.rows == 1 else 128 * self.cols


def _validate(d):
    if d.rows < 1 or d.cols < 0 or d.g < 1:
        raise ValueError("bad tensor shape or granularity")
    if d.adam_kind == ADAM_FLAT256:
        if d.g % 256:
            raise ValueError("flat 256-element Adam blocks need g % 256 == 0")
    elif d.adam_kind == ADAM_TILE128:
        if d.g % d.tile_unit():
            raise ValueError("128x128 Adam tiles need g to be whole 128-row bands")
    elif d.adam_kind == ADAM_TILE32:
        if d.g % (32 if d.rows == 1 else 32 * d.cols) or d.fp8:
            raise ValueError("32x32 Adam tiles need g to be whole 32-row bands and take no FP8 staging")
    elif d.adam_kind == OPT_MUON:
        if d.rows < 2 or d.fp8:
            raise ValueError("Muon tensors are 2-D and take no FP8 staging")
    else:
        raise ValueError("unknown Adam block kind")
    if d.fp8 and d.g % d.tile_unit():
        raise ValueError("128x128 FP8 tiles need g to be whole 128-row bands")


def tiles_in(d, length):
    """Number of 128x128 tiles (1-D: 1x128) covering ``length`` elements of d that
    start on a band boundary."""
    if d.rows == 1:
        return -(-length // 128)
    rows = length // d.cols
    return -(-rows // 128) * -(-d.cols // 128)


def tiles32_in(d, length):
    """32x32 tiles (1-D: 32-element blocks) covering ``length`` elements of d that
    start on a 32-row band boundary."""
    if d.rows == 1:
        return -(-length // 32)
    rows = length // d.cols
    return -(-rows // 32) * -(-d.cols // 32)


def adam_blocks_in(d, length):
    if d.adam_kind == OPT_MUON:
        return 0
    if d.adam_kind == ADAM_TILE32:
        return tiles32_in(d, length)
    if d.adam_kind == ADAM_FLAT256:
        return -(-length // 256)
    return tiles_in(d, length)


class Layout:
    """Planned DBuffer layout plus the derived tables.

    intervals: list of (dev, tensor, t_off, len, local_off, mslot, fslot) in device
    order, tensors in buffer order within a device.  mslot / fslot are global slot
    numbers of the interval's first Adam block / FP8 tile (fslot = -1 without FP8);
    slots are numbered per device in interval order and, inside an interval, in
    tensor-flat order for 256-element blocks and band-major, column-tile-minor order
    for 128x128 tiles.  dev_table[k] = (first interval, mslot base, fslot base) for
    k = 0..V (entry V closes the ranges)."""

    def __init__(self, descs, V, S, starts):
        self.descs, self.V, self.S, self.starts = descs, V, S, starts
        order = sorted(range(len(descs)), key=lambda i: starts[i])
        self.intervals, self.dev_table = [], []
        mslot = fslot = 0
        for k in range(V):
            self.dev_table.append((len(self.intervals), mslot, fslot))
            lo_k, hi_k = k * S, (k + 1) * S
            for i in order:
                d = descs[i]
                lo = max(starts[i], lo_k)
                hi = min(starts[i] + d.numel, hi_k)
                if hi <= lo:
                    continue
                t_off, ln = lo - starts[i], hi - lo
                fs = fslot if d.fp8 else -1
                self.intervals.append((k, i, t_off, ln, lo - lo_k, mslot, fs))
                mslot += adam_blocks_in(d, ln)
                if d.fp8:
                    fslot += tiles_in(d, ln)
        self.dev_table.append((len(self.intervals), mslot, fslot))
        self.n_mslots, self.n_fslots = mslot, fslot

    def export(self):
        """Flat int64 table:
        header   [magic, version, V, S, N, NI, n_mslots, n_fslots]
        tensors  N  x [start, numel, rows, cols, g, adam_kind, fp8]
        intervals NI x [dev, tensor, t_off, len, local_off, mslot, fslot]
        devices  (V+1) x [first interval, mslot base, fslot base]"""
        out = [EXPORT_MAGIC, EXPORT_VERSION, self.V, self.S, len(self.descs),
               len(self.intervals), self.n_mslots, self.n_fslots]
        for i, d in enumerate(self.descs):
            out += [self.starts[i], d.numel, d.rows, d.cols, d.g, d.adam_kind, int(d.fp8)]
        for iv in self.intervals:
            out += list(iv)
        for row in self.dev_table:
            out += list(row)
        return out

    def total_elems(self):
        return sum(d.numel for d in self.descs)

    def padding_fraction(self):
        return 1.0 - self.total_elems() / (self.V * self.S)


ORDER_GIVEN, ORDER_BLOCK, ORDER_SHAPE = 0, 1, 2


def placement_order(descs, kind=ORDER_GIVEN):
    """The orders the walkthrough (paper section 5) says were tried: as given (the
    default), sorted by block size, sorted by tensor shape.  Readings: block size
    = atomic granularity g, largest first; shape = (rows, cols), largest first,
    so equal shapes sit together; ties keep the given order."""
    idx = list(range(len(descs)))
    if kind == ORDER_GIVEN:
        return idx
    if kind == ORDER_BLOCK:
        return sorted(idx, key=lambda i: (-descs[i].g, i))
    if kind == ORDER_SHAPE:
        return sorted(idx, key=lambda i: (-descs[i].rows, -descs[i].cols, i))
    raise ValueError("unknown order")


def plan(descs, V, alpha=128, start_align=16, order=ORDER_GIVEN):
    """Validate the descriptors, run the heuristic, build the derived tables."""
    for d in descs:
        _validate(d)
    S, starts, _ = plan_sizes([d.numel for d in descs], [d.g for d in descs], V, alpha, start_align,
                              placement_order(descs, order))
    return Layout(descs, V, S, starts)


# ----------------------------------------------------------------------------- block enumeration


def adam_blocks(layout, dev_lo, dev_hi):
    """Yield (slot index relative to dev_lo's first slot, local element positions)
    for every Adam block of devices [dev_lo, dev_hi).  Local positions index a
    buffer that starts at global offset dev_lo * S."""
    yield from _blocks(layout, dev_lo, dev_hi, fp8=False)


def fp8_tiles(layout, dev_lo, dev_hi):
    """Same for FP8 tiles (tensors without FP8 yield nothing)."""
    yield from _blocks(layout, dev_lo, dev_hi, fp8=True)


def _blocks(layout, dev_lo, dev_hi, fp8):
    S = layout.S
    first, _, _ = layout.dev_table[dev_lo]
    last, _, _ = layout.dev_table[dev_hi]
    base = layout.dev_table[dev_lo][2 if fp8 else 1]
    for (k, i, t_off, ln, loff, mslot, fslot) in layout.intervals[first:last]:
        d = layout.descs[i]
        if (fp8 and not d.fp8) or (not fp8 and d.adam_kind == OPT_MUON):
            continue
        slot = (fslot if fp8 else mslot) - base
        pos0 = (k - dev_lo) * S + loff - t_off  # local position of tensor element 0
        if not fp8 and d.adam_kind == ADAM_FLAT256:
            for f in range(t_off, t_off + ln, 256):
                yield slot, pos0 + range_array(f, min(f + 256, t_off + ln))
                slot += 1
        elif not fp8 and d.adam_kind == ADAM_TILE32:
            yield from _tiles(d, t_off, ln, pos0, slot, 32)
        elif d.rows == 1:
            for f in range(t_off, t_off + ln, 128):
                yield slot, pos0 + range_array(f, min(f + 128, t_off + ln))
                slot += 1
        else:
            C = d.cols
            r0, r1 = t_off // C, (t_off + ln) // C
            for rb in range(r0, r1, 128):
                rows = range_array(rb, min(rb + 128, r1))
                for cb in range(0, C, 128):
                    cols = range_array(cb, min(cb + 128, C))
                    yield slot, pos0 + (rows[:, None] * C + cols[None, :]).ravel()
                    slot += 1


def _tiles(d, t_off, ln, pos0, slot, T):
    """T x T tiles (1-D: T-element blocks) of the interval, band-major,
    column-tile-minor, clipped at the tensor's edges."""
    if d.rows == 1:
        for f in range(t_off, t_off + ln, T):
            yield slot, pos0 + range_array(f, min(f + T, t_off + ln))
            slot += 1
        return
    C = d.cols
    r0, r1 = t_off // C, (t_off + ln) // C
    for rb in range(r0, r1, T):
        rows = range_array(rb, min(rb + T, r1))
        for cb in range(0, C, T):
            cols = range_array(cb, min(cb + T, C))
            yield slot, pos0 + (rows[:, None] * C + cols[None, :]).ravel()
            slot += 1


def block_at(layout, dev_lo, dev_hi, pos, fp8=False):
    """(slot, local positions) of the Adam block (or FP8 tile) holding local
    position ``pos`` of shards [dev_lo, dev_hi), or None for padding / a tensor
    without FP8.  Same slot rules as _blocks, for one block."""
    S = layout.S
    k = dev_lo + pos // S
    loff_in = pos - (k - dev_lo) * S
    first, _, _ = layout.dev_table[k]
    last, _, _ = layout.dev_table[k + 1]
    base = layout.dev_table[dev_lo][2 if fp8 else 1]
    for (kk, i, t_off, ln, loff, mslot, fslot) in layout.intervals[first:last]:
        if not (loff <= loff_in < loff + ln):
            continue
        d = layout.descs[i]
        if (fp8 and not d.fp8) or (not fp8 and d.adam_kind == OPT_MUON):
            return None
        slot0 = (fslot if fp8 else mslot) - base
        pos0 = (k - dev_lo) * S + loff - t_off
        f = t_off + (loff_in - loff)  # tensor-flat offset
        if not fp8 and d.adam_kind == ADAM_FLAT256:
            j = (f - t_off) // 256
            a = t_off + 256 * j
            return slot0 + j, pos0 + range_array(a, min(a + 256, t_off + ln))
        T = 32 if (not fp8 and d.adam_kind == ADAM_TILE32) else 128
        if d.rows == 1:
            j = (f - t_off) // T
            a = t_off + T * j
            return slot0 + j, pos0 + range_array(a, min(a + T, t_off + ln))
        C = d.cols
        r0, r1 = t_off // C, (t_off + ln) // C
        r, c = f // C, f % C
        band, ct = (r - r0) // T, c // T
        nct = -(-C // T)
        rows = range_array(r0 + T * band, min(r0 + T * band + T, r1))
        cols = range_array(T * ct, min(T * ct + T, C))
        return slot0 + band * nct + ct, pos0 + (rows[:, None] * C + cols[None, :]).ravel()
    return None


def range_array(a, b):
    return np.arange(a, b, dtype=np.int64)
