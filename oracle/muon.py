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
