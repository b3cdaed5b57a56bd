"""Muon's Newton-Schulz orthogonalisation on a whole matrix, in fp64 (oracle; test
infrastructure only).

Source: feynmanwiki walkthrough of veScale-FSDP, paper section 6.3 (the Muon
experiment): Muon's matrix-sign preconditioner needs the complete 2-D matrix; the
momentum matrix is redistributed to one load-balanced root, which runs the
Newton-Schulz iteration and sends the result back.  The pages give neither the
iteration nor its coefficients.

Reading: the quintic Newton-Schulz iteration
    X <- X / (||X||_F + eps)
    repeat steps times:  A = X X^T;  B = b A + c A A;  X = a X + B X
with (a, b, c) = (3.4445, -4.7750, 2.0315), 5 steps, eps = 1e-7; a tall input
(rows > cols) is iterated as its transpose and transposed back.  Each step maps
every singular value x of X to a x + b x^3 + c x^5 and keeps the singular vectors.
"""

import numpy as np

NS_A, NS_B, NS_C = 3.4445, -4.7750, 2.0315


def newton_schulz(x, steps=5, a=NS_A, b=NS_B, c=NS_C, eps=1e-7):
    """x: 2-D array (any float dtype).  Returns the fp64 result, same shape."""
    X = np.array(x, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = X / (np.linalg.norm(X) + eps)
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if tall else X


# ----------------------------------------------------------------------------- the Muon step around it
# Same passage (paper section 6.3 in the walkthrough): each 2-D weight W gets its
# gradient G, the momentum update produces M, a load-balanced root is chosen, the
# full M materialises only on that root, the root runs Newton-Schulz, and the
# result goes back to W's placement, where it is applied to W.  The pages print
# no formula for any of these steps.
#
# Readings (the plainest ones the passage supports):
#   momentum   M <- fma(mu, M, G) in fp32 (heavy-ball momentum, one rounding)
#   root       longest-processing-time greedy on the Newton-Schulz cost
#              4 m^2 n + 2 m^3 (m = min dim, n = max dim): matrices by cost,
#              largest first (ties: lower tensor index), each to the device with
#              the least assigned cost so far (ties: lower device index)
#   NS input   M rounded to bf16 (round to nearest even), row-major full matrix
#   apply      W <- fma(-lr, O, W) in fp32, O the bf16 Newton-Schulz output

from .codecs import bf16_bits_to_f32, f32_to_bf16_bits, fma32  # noqa: E402
from .planner import OPT_MUON  # noqa: E402


def ns_cost(rows, cols):
    """Nominal flops of one Newton-Schulz step on a rows x cols matrix."""
    m, n = min(rows, cols), max(rows, cols)
    return 4 * m * m * n + 2 * m ** 3


def muon_roots(descs, V):
    """Root device of every Muon tensor (-1 for the others)."""
    roots = [-1] * len(descs)
    muon = [i for i, d in enumerate(descs) if d.adam_kind == OPT_MUON]
    muon.sort(key=lambda i: (-ns_cost(descs[i].rows, descs[i].cols), i))
    load = [0] * V
    for i in muon:
        k = min(range(V), key=lambda j: (load[j], j))
        roots[i] = k
        load[k] += ns_cost(descs[i].rows, descs[i].cols)
    return roots


def _muon_pieces(layout, dev_lo, dev_hi):
    """(local position, tensor, t_off, len) of every Muon interval in the range."""
    first, _, _ = layout.dev_table[dev_lo]
    last, _, _ = layout.dev_table[dev_hi]
    for (k, i, t_off, ln, loff, _, _) in layout.intervals[first:last]:
        if layout.descs[i].adam_kind == OPT_MUON:
            yield (k - dev_lo) * layout.S + loff, i, t_off, ln


def muon_momentum(layout, dev_lo, dev_hi, grad_bits, mom, mu):
    """One momentum update over local shards [dev_lo, dev_hi).
    grad_bits: bf16 gradient DBuffer (uint16); mom: fp32 momentum DBuffer.
    Returns (new mom, {tensor: (t_off, bf16 bits of M over that range)...} as a
    list of pieces per tensor)."""
    mom = np.array(mom, dtype=np.float32, copy=True)
    gathered = {}
    mu32 = np.float32(mu)
    for pos, i, t_off, ln in _muon_pieces(layout, dev_lo, dev_hi):
        sl = slice(pos, pos + ln)
        g = bf16_bits_to_f32(grad_bits[sl])
        m = fma32(np.full(ln, mu32), mom[sl], g)
        mom[sl] = m
        gathered.setdefault(i, []).append((t_off, f32_to_bf16_bits(m)))
    return mom, gathered


def assemble(desc, pieces):
    """Full row-major bf16 matrix (uint16) of one tensor from its gathered pieces
    (every element must be covered exactly once)."""
    out = np.zeros(desc.rows * desc.cols, np.uint16)
    seen = np.zeros(desc.rows * desc.cols, bool)
    for t_off, bits in pieces:
        assert not seen[t_off:t_off + len(bits)].any()
        out[t_off:t_off + len(bits)] = bits
        seen[t_off:t_off + len(bits)] = True
    assert seen.all()
    return out.reshape(desc.rows, desc.cols)


def muon_apply(layout, dev_lo, dev_hi, master, updates, lrs):
    """W <- fma(-lr_i, O_i, W) on every Muon interval in the range.
    updates: {tensor: full row-major bf16 bits (uint16) of O}; lrs: {tensor: lr}."""
    master = np.array(master, dtype=np.float32, copy=True)
    for pos, i, t_off, ln in _muon_pieces(layout, dev_lo, dev_hi):
        if i not in updates:
            continue
        sl = slice(pos, pos + ln)
        o = bf16_bits_to_f32(np.asarray(updates[i]).reshape(-1)[t_off:t_off + ln])
        master[sl] = fma32(np.full(ln, -np.float32(lrs[i])), o, master[sl])
    return master
