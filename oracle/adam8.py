"""Block-wise 8-bit Adam on the local DBuffer shard (oracle; test infrastructure
only).

Sources: "veScale-FSDP: Flexible and High-Performance FSDP at Scale" (bud-325
summary), Key claims: RaggedShard's block granularity supports 8-bit Adam, i.e.
block-quantised optimizer state; feynmanwiki walkthrough, paper section 6.3 (the
8-bit Adam experiment): the optimizer statistics are quantised per block, every
quantisation block stays inside one local shard, so each device requantises its
own state with no exchange of scale metadata.

Readings (the pages give neither the update nor the quantiser):
  * Adam without weight decay; the update uses the fp32 values m', v' computed in
    this step, only their storage is 8-bit;
  * m is stored as int8 codes in [-127, 127] and v as uint8 codes, each block with
    one fp32 absmax scale (linear map, see codecs.quant_*_absmax);
  * the per-element order of operations is fixed, each step one IEEE fp32
    operation rounded to nearest; fma(x, y, z) = x*y + z rounded once:
        g   = f32(bf16 grad)
        m   = code_m * s_m            v   = code_v * s_v
        m'  = fma(b1, m, omb1*g)      v'  = fma(b2, v, omb2*(g*g))
        mh  = m' * rbc1               vh  = v' * rbc2
        u   = mh / (sqrt(vh) + eps)   p'  = fma(-lr, u, p)
    with omb1 = 1-b1, omb2 = 1-b2 and the reciprocal bias corrections
    rbc1 = 1/(1-b1^t), rbc2 = 1/(1-b2^t) evaluated in fp64 and rounded once to
    fp32 (adam_hparams);
  * a block is 256 consecutive elements of the tensor (the last one may be short),
    or a 128x128 tile of the tensor's 2-D view (1-D tensors: 128 elements).
"""

import numpy as np

from .codecs import bf16_bits_to_f32, dequant, fma32, quant_int8_absmax, quant_uint8_absmax
from .planner import adam_blocks

F32 = np.float32


def adam_hparams(lr, b1, b2, eps, t):
    """fp32 hyper-parameters, the derived ones computed in fp64 then rounded."""
    lr, b1, b2, eps = float(lr), float(b1), float(b2), float(eps)
    return dict(lr=F32(lr), b1=F32(b1), b2=F32(b2), eps=F32(eps),
                omb1=F32(1.0 - b1), omb2=F32(1.0 - b2),
                rbc1=F32(1.0 / (1.0 - b1 ** t)), rbc2=F32(1.0 / (1.0 - b2 ** t)))


def adam_update(g_bits, p, m, v, hp):
    """Elementwise fp32 Adam update from dequantised state.  Returns (p', m', v')."""
    g = bf16_bits_to_f32(g_bits)
    p = np.asarray(p, dtype=np.float32)
    m1 = fma32(hp["b1"], m, hp["omb1"] * g)
    v1 = fma32(hp["b2"], v, hp["omb2"] * (g * g))
    mh = m1 * hp["rbc1"]
    vh = v1 * hp["rbc2"]
    u = mh / (np.sqrt(vh) + hp["eps"])
    p1 = fma32(-hp["lr"], u, p)
    return p1.astype(np.float32), m1.astype(np.float32), v1.astype(np.float32)


def adam8_block(g_bits, p, qm, qv, sm, sv, hp):
    """One quantisation block: dequantise, update, requantise.
    Returns (p', codes_m', codes_v', s_m', s_v')."""
    m = dequant(qm, sm)
    v = dequant(qv, sv)
    p1, m1, v1 = adam_update(g_bits, p, m, v, hp)
    qm1, sm1 = quant_int8_absmax(m1)
    qv1, sv1 = quant_uint8_absmax(v1)
    return p1, qm1, qv1, sm1, sv1


def adam8_step(layout, dev_lo, dev_hi, grad, master, m, v, m_scale, v_scale, hp, blocks=None):
    """Apply adam8_block to every Adam block of local shards [dev_lo, dev_hi) (or to
    the given subset of (slot, positions) pairs).  Arrays index the local buffer
    starting at global offset dev_lo*S; scales index slots relative to dev_lo's
    first slot.  Returns updated copies (master, m, v, m_scale, v_scale); padding
    is left untouched."""
    master, m, v = master.copy(), m.copy(), v.copy()
    m_scale, v_scale = m_scale.copy(), v_scale.copy()
    it = adam_blocks(layout, dev_lo, dev_hi) if blocks is None else blocks
    for slot, pos in it:
        p1, qm1, qv1, sm1, sv1 = adam8_block(grad[pos], master[pos], m[pos], v[pos],
                                             m_scale[slot], v_scale[slot], hp)
        master[pos], m[pos], v[pos] = p1, qm1, qv1
        m_scale[slot], v_scale[slot] = sm1, sv1
    return master, m, v, m_scale, v_scale
