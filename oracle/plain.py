"""Plain-definition leg of the 8-bit Adam step and the FP8 requantisation
(oracle; test infrastructure only).

The pages ("veScale-FSDP: Flexible and High-Performance FSDP at Scale", Key
claims: 8-bit Adam and block-wise FP8 on RaggedShard blocks; the feynmanwiki
walkthrough, paper section 6.3) fix the method - Adam with per-block quantised
state, block-wise FP8 of the updated parameters - but no order of floating-point
operations.  The contract leg (``adam8``, ``fp8``, ``codecs``) states one order,
chosen to match the kernels' instruction form: fused multiply-adds in the moment
updates and the parameter step, reciprocal bias corrections, and codes from the
product with a reciprocal block scale.  This module restates the same method in
the plainest order instead, so that the distance between the kernels and the
textbook definition can be measured:

    g   = f32(bf16 grad)                    m = code_m * s_m,  v = code_v * s_v
    m'  = b1*m + omb1*g                     v' = b2*v + omb2*(g*g)
    mh  = m' / bc1                          vh = v' / bc2
    p'  = p - lr * (mh / (sqrt(vh) + eps))
    block state:  s = amax / qmax,  code = clamp(rint(fp32(x / s)))   (s == 0: codes 0)
    FP8 tile:     s = amax / 448,   code = e4m3(fp32(p' / s))          (s == 0: +-0)

every operation one IEEE fp32 operation rounded to nearest (ties to even), no
fused operation anywhere; omb = 1 - b and bc = 1 - b^t evaluated in fp64 and
rounded once to fp32.  The number formats (bf16, E4M3 encode / decode) are the
ones ``codecs`` defines; nothing else is shared with the contract leg.
"""

import numpy as np

from .codecs import bf16_bits_to_f32, e4m3_encode
from .planner import adam_blocks, fp8_tiles

F32 = np.float32


def adam_hparams(lr, b1, b2, eps, t):
    """fp32 hyper-parameters with the bias corrections themselves (not their
    reciprocals): bc = 1 - b^t in fp64, rounded once."""
    lr, b1, b2, eps = float(lr), float(b1), float(b2), float(eps)
    return dict(lr=F32(lr), b1=F32(b1), b2=F32(b2), eps=F32(eps), omb1=F32(1.0 - b1), omb2=F32(1.0 - b2),
                bc1=F32(1.0 - b1 ** t), bc2=F32(1.0 - b2 ** t))


def adam_update(g_bits, p, m, v, hp):
    """Elementwise fp32 Adam update, every multiply, add, division and square
    root a separate rounded operation.  Returns (p', m', v')."""
    g = bf16_bits_to_f32(g_bits)
    p = np.asarray(p, dtype=np.float32)
    m = np.asarray(m, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    m1 = hp["b1"] * m + hp["omb1"] * g
    v1 = hp["b2"] * v + hp["omb2"] * (g * g)
    mh = m1 / hp["bc1"]
    vh = v1 / hp["bc2"]
    step = hp["lr"] * (mh / (np.sqrt(vh) + hp["eps"]))
    p1 = p - step
    return p1.astype(np.float32), m1.astype(np.float32), v1.astype(np.float32)


def _quant(x, amax, qmax, lo, hi, dtype):
    s = F32(amax) / F32(qmax)
    if s == 0:
        return np.zeros(x.shape, dtype), F32(0)
    q = np.rint(x / s)  # fp32 quotient, then half-to-even
    return np.clip(q, lo, hi).astype(dtype), F32(s)


def quant_int8(x):
    """Signed block: s = max|x| / 127, code = clamp(rint(fp32(x / s)), -127, 127)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.max(np.abs(x)) if x.size else F32(0)
    return _quant(x, amax, 127, -127, 127, np.int8)


def quant_uint8(x):
    """Non-negative block: s = max x / 255, code = clamp(rint(fp32(x / s)), 0, 255)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.max(x) if x.size else F32(0)
    return _quant(x, amax, 255, 0, 255, np.uint8)


def fp8_tile(p):
    """One FP8 tile: s = max|p| / 448, code = e4m3(fp32(p / s)); s == 0 keeps
    each element's sign on a zero code."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    amax = np.max(np.abs(p)) if p.size else F32(0)
    s = F32(amax) / F32(448)
    if s == 0:
        return (p.view(np.uint32) >> 24).astype(np.uint8) & np.uint8(0x80), F32(0)
    return e4m3_encode(p / s), F32(s)


def adam8_block(g_bits, p, qm, qv, sm, sv, hp):
    """One block: dequantise (code * scale), update, requantise."""
    m = np.asarray(qm).astype(np.float32) * F32(sm)
    v = np.asarray(qv).astype(np.float32) * F32(sv)
    p1, m1, v1 = adam_update(g_bits, p, m, v, hp)
    qm1, sm1 = quant_int8(m1)
    qv1, sv1 = quant_uint8(v1)
    return p1, qm1, qv1, sm1, sv1


def adam8_step(layout, dev_lo, dev_hi, grad, master, m, v, m_scale, v_scale, hp):
    """adam8_block over every Adam block of local shards [dev_lo, dev_hi); the
    same buffers and slots as the contract leg.  Returns updated copies."""
    master, m, v = master.copy(), m.copy(), v.copy()
    m_scale, v_scale = m_scale.copy(), v_scale.copy()
    for slot, pos in adam_blocks(layout, dev_lo, dev_hi):
        p1, qm1, qv1, sm1, sv1 = adam8_block(grad[pos], master[pos], m[pos], v[pos], m_scale[slot], v_scale[slot], hp)
        master[pos], m[pos], v[pos] = p1, qm1, qv1
        m_scale[slot], v_scale[slot] = sm1, sv1
    return master, m, v, m_scale, v_scale


def quant_fp8(layout, dev_lo, dev_hi, master, fp8_out, fp8_scale):
    """fp8_tile over every FP8 tile of local shards [dev_lo, dev_hi)."""
    fp8_out, fp8_scale = fp8_out.copy(), fp8_scale.copy()
    for slot, pos in fp8_tiles(layout, dev_lo, dev_hi):
        q, s = fp8_tile(master[pos])
        fp8_out[pos] = q
        fp8_scale[slot] = s
    return fp8_out, fp8_scale
