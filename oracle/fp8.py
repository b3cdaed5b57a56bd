"""Block-wise FP8 requantisation of updated parameters into the AllGather staging
buffer (oracle; test infrastructure only).

Sources: "veScale-FSDP: Flexible and High-Performance FSDP at Scale" (bud-325
summary), TL;DR and Key claims: block-wise FP8 in the DeepSeek-V3 style, one
scale per block; feynmanwiki walkthrough (paper sections 2-4): every quantisation
block must live entirely on one device because its values share scale metadata,
which is what RaggedShard's granularity guarantees.

Readings (the pages give no formula): blocks are 128x128 tiles of the tensor's
row-major 2-D view, clipped at the edges (1-D tensors: 1x128); per tile
    amax = max |p'|,  s = amax / 448 (fp32 division, the stored scale),
    r = 448 / amax (fp32 division, once per tile),
    code = e4m3(p' * r)  (fp32 product, then round-to-nearest-even, saturating),
(p' / s instead when r overflows, amax below ~1.3e-36), and a tile whose scale
is 0 gets s = 0 with codes +0 / -0 following each element's sign.
Codes go to the same local offsets as the parameters; s goes to the tile's slot.
"""

import numpy as np

from .codecs import block_scale, e4m3_encode, scaled
from .planner import fp8_tiles

F32 = np.float32


def fp8_tile(p):
    """One tile -> (uint8 E4M3 codes, fp32 scale)."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    amax = np.max(np.abs(p)) if p.size else F32(0)
    s, r, mode = block_scale(amax, 448)
    if mode == 0:  # +-0 codes following each element's sign
        return (p.view(np.uint32) >> 24).astype(np.uint8) & np.uint8(0x80), F32(0)
    return e4m3_encode(scaled(p, s, r, mode)), s


def quant_fp8(layout, dev_lo, dev_hi, master, fp8_out, fp8_scale, tiles=None):
    """Requantise every FP8 tile of local shards [dev_lo, dev_hi) (or the given
    subset).  Returns updated copies (fp8_out, fp8_scale); bytes outside tiles are
    left as they were."""
    fp8_out, fp8_scale = fp8_out.copy(), fp8_scale.copy()
    it = fp8_tiles(layout, dev_lo, dev_hi) if tiles is None else tiles
    for slot, pos in it:
        q, s = fp8_tile(master[pos])
        fp8_out[pos] = q
        fp8_scale[slot] = s
    return fp8_out, fp8_scale


# ----------------------------------------------------------------------------- the view after the AllGather
# Same sources: the gathered FP8 buffer serves the forward and backward compute,
# which (DeepSeek-V3 style) reads each parameter as code x tile scale.  Reading
# (the pages give no formula): the E4M3 code decoded exactly, times the tile's
# fp32 scale in fp32 (one rounding), then rounded to bf16 (nearest even); only
# FP8 tensors are written, every other element of the output is left as it was.

def dequant_tile(q, s):
    """uint8 E4M3 codes and the tile's fp32 scale -> bf16 bits (uint16)."""
    from .codecs import e4m3_decode, f32_to_bf16_bits

    x = e4m3_decode(np.asarray(q, np.uint8)).astype(np.float32) * F32(s)
    return f32_to_bf16_bits(x.astype(np.float32))


def dequant_fp8(layout, dev_lo, dev_hi, fp8, fp8_scale, out_bf16):
    """bf16 view of every FP8 tile of local shards [dev_lo, dev_hi); returns an
    updated copy of out_bf16 (uint16)."""
    out = np.array(out_bf16, dtype=np.uint16, copy=True)
    for slot, pos in fp8_tiles(layout, dev_lo, dev_hi):
        out[pos] = dequant_tile(fp8[pos], fp8_scale[slot])
    return out
