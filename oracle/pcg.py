"""Oracle for Jacobi-preconditioned conjugate gradients (numpy, fp64, CPU).

TEST INFRASTRUCTURE ONLY, like the rest of this package.

Source: "Fused FEM matvec" page, section 6.1: the solver around the
matrix-vector products is CG with the Jacobi (diagonal) preconditioner,
whose iteration count grows like the square root of the condition number.
The page does not print the recurrence; this is the textbook preconditioned
CG, step by step:

    r = b - A x;  z = D^-1 r;  p = z;  rz = r.z
    repeat:  q = A p;  alpha = rz / (p.q);  x += alpha p;  r -= alpha q
             stop when ||r|| <= tol ||b||
             z = D^-1 r;  rz' = r.z;  beta = rz' / rz;  rz = rz';  p = z + beta p

with D the diagonal of A (a zero diagonal entry leaves its row unscaled).
The stopping test is on the recurrence's residual r, as in the library.
"""
from __future__ import annotations

import numpy as np


def jacobi_pcg(matvec, diag, b, x0, tol: float, max_iter: int):
    """Returns (x, iterations, status, residual norms ||r_k|| for k = 0..),
    status 1 converged, 2 iteration limit, 3 breakdown."""
    d = np.asarray(diag, dtype=np.float64)
    dinv = np.where(d != 0.0, 1.0 / np.where(d != 0.0, d, 1.0), 1.0)
    b = np.asarray(b, dtype=np.float64)
    x = np.asarray(x0, dtype=np.float64).copy()
    r = b - matvec(x)
    z = dinv * r
    p = z.copy()
    rz = r @ z
    bnorm = np.sqrt(b @ b)
    hist = [np.sqrt(r @ r)]
    if hist[-1] <= tol * bnorm:
        return x, 0, 1, hist
    if max_iter <= 0:
        return x, 0, 2, hist
    for it in range(1, max_iter + 1):
        q = matvec(p)
        pq = p @ q
        if not pq > 0.0:
            return x, it - 1, 3, hist
        alpha = rz / pq
        x += alpha * p
        r -= alpha * q
        hist.append(np.sqrt(r @ r))
        if hist[-1] <= tol * bnorm:
            return x, it, 1, hist
        z = dinv * r
        rz_new = r @ z
        beta = rz_new / rz
        rz = rz_new
        p = z + beta * p
    return x, max_iter, 2, hist
