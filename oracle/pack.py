"""Group-level fused pre-communication op into the gradient DBuffer (oracle; test
infrastructure only).

Source: "veScale-FSDP: Flexible and High-Performance FSDP at Scale" (bud-325
summary), Key claims and Method: DBuffer fuses the identical per-tensor
pre-communication kernels (add / scale / zero / copy) at group level; the
feynmanwiki walkthrough (paper section 5, DBuffer paragraphs) adds that each tensor
is a view of its planned slice so the collective then runs on the buffer in place.

Reading (the pages give no formula): for every element j of every interval of the
local shards [dev_lo, dev_hi),
    y = f32(grad_i[t_off + j]) * scale                      (copy + scale)
    y = f32(dbuf[pos]) + y            only with accumulate  (add)
    dbuf[pos] = bf16_rne(y)
and every padding element of those shards is set to +0 (zero).  Each arithmetic
step is one IEEE fp32 operation rounded to nearest.
"""

import numpy as np

from .codecs import bf16_bits_to_f32, f32_to_bf16_bits


def pack(layout, dev_lo, dev_hi, grads, dbuf, scale, accumulate):
    """grads[i] = (bits, base): uint16 bf16 bits of tensor i holding tensor-flat
    elements [base, base + len(bits)).  dbuf: uint16 bf16 bits of the local shards
    [dev_lo, dev_hi) (length (dev_hi - dev_lo) * S).  Returns the new dbuf."""
    S = layout.S
    dbuf = np.asarray(dbuf, dtype=np.uint16)
    assert dbuf.shape == ((dev_hi - dev_lo) * S,)
    out = np.zeros_like(dbuf)  # padding := +0
    sc = np.float32(scale)
    first, _, _ = layout.dev_table[dev_lo]
    last, _, _ = layout.dev_table[dev_hi]
    for (k, i, t_off, ln, loff, _, _) in layout.intervals[first:last]:
        bits, base = grads[i]
        src = bf16_bits_to_f32(bits[t_off - base:t_off - base + ln])
        y = src * sc
        pos = (k - dev_lo) * S + loff
        if accumulate:
            y = bf16_bits_to_f32(dbuf[pos:pos + ln]) + y
        out[pos:pos + ln] = f32_to_bf16_bits(y)
    return out


def unpack(layout, dev_lo, dev_hi, dbuf):
    """Inverse view: tensor i -> (bits of its owned range, base) read back from the
    buffer.  Used by the round-trip pin."""
    S = layout.S
    first, _, _ = layout.dev_table[dev_lo]
    last, _, _ = layout.dev_table[dev_hi]
    parts = {}
    for (k, i, t_off, ln, loff, _, _) in layout.intervals[first:last]:
        pos = (k - dev_lo) * S + loff
        parts.setdefault(i, []).append((t_off, dbuf[pos:pos + ln]))
    out = {}
    for i, segs in parts.items():
        segs.sort(key=lambda t: t[0])
        base = segs[0][0]
        out[i] = (np.concatenate([s for _, s in segs]), base)
    return out
