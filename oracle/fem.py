"""Oracle for the matrix-free stiffness operator y = K x on a structured hex
mesh (numpy, fp64, CPU).

TEST INFRASTRUCTURE ONLY, like the rest of this package.

Source: "Fused FEM matvec" page (bbs.csdn.net), section 2.1: y = K x without
storing K, as three steps per element -- gather the element's 24 dofs from x
through the element-to-dof table, multiply by the 24 x 24 element matrix,
scatter-add the 24 results into y; section 5.2: with a uniform material all
elements share one matrix (kept in constant memory), here scaled by the
element's density as in the page's SIMP setting.

Readings (each also in the design notes):

* Element e = ex + nex*(ey + ney*ez) of an nex x ney x nez mesh; node
  (i, j, k) = i + (nex+1)*(j + (ney+1)*k); dof = 3*node + c. Element e's local
  node b sits at (ex, ey, ez) + H[b] with H the corner order (0,0,0), (1,0,0),
  (1,1,0), (0,1,0), (0,0,1), (1,0,1), (1,1,1), (0,1,1) (bottom face
  anticlockwise, then the top face); local dof 3*b + c.
* Ke = rho_e * K0, so y = sum_e P_e^T (rho_e K0 (P_e x)).
* ``s`` (the scale of the parity tolerance) sums |rho_e K0[a, j] x[dof_j]|
  over every element term that lands in a dof, because the operator adds the
  element terms one by one and never forms the assembled entries.
"""
from __future__ import annotations

import numpy as np

from . import csr_spmv

CORNERS = np.array([(0, 0, 0), (1, 0, 0), (1, 1, 0), (0, 1, 0),
                    (0, 0, 1), (1, 0, 1), (1, 1, 1), (0, 1, 1)], dtype=np.int64)


def element_dofs(nex: int, ney: int, nez: int) -> np.ndarray:
    """int64[n_elem, 24]: the global dof of each element's local dof."""
    e = np.arange(nex * ney * nez, dtype=np.int64)
    ex, ey, ez = e % nex, (e // nex) % ney, e // (nex * ney)
    i = ex[:, None] + CORNERS[None, :, 0]
    j = ey[:, None] + CORNERS[None, :, 1]
    k = ez[:, None] + CORNERS[None, :, 2]
    node = i + (nex + 1) * (j + (ney + 1) * k)                       # [E, 8]
    return (3 * node[:, :, None] + np.arange(3)[None, None, :]).reshape(-1, 24)


def fem_matvec(nex, ney, nez, rho, K0, x, with_abs: bool = True):
    """y = sum_e P_e^T (rho_e K0 (P_e x)) in fp64, element by element: gather,
    local product, scatter-add (and s, the sum of the terms' magnitudes)."""
    edof = element_dofs(nex, ney, nez)
    n_dofs = 3 * (nex + 1) * (ney + 1) * (nez + 1)
    r = np.asarray(rho, dtype=np.float64)
    k0 = np.asarray(K0, dtype=np.float64)
    xv = np.asarray(x, dtype=np.float64)
    u = xv[edof]                                           # gather   [E, 24]
    f = r[:, None] * (u @ k0.T)                            # Ke u     [E, 24]
    y = np.zeros(n_dofs)
    np.add.at(y, edof.reshape(-1), f.reshape(-1))          # scatter-add
    if not with_abs:
        return y
    fa = np.abs(r)[:, None] * (np.abs(u) @ np.abs(k0).T)
    s = np.zeros(n_dofs)
    np.add.at(s, edof.reshape(-1), fa.reshape(-1))
    return y, s


def fem_assemble(nex, ney, nez, rho, K0):
    """The assembled K (CSR, fp64 values, columns sorted within a row): every
    element adds rho_e K0[a, b] at (dof_a, dof_b)."""
    edof = element_dofs(nex, ney, nez)
    n_dofs = 3 * (nex + 1) * (ney + 1) * (nez + 1)
    r = np.asarray(rho, dtype=np.float64)
    k0 = np.asarray(K0, dtype=np.float64)
    rows = np.repeat(edof, 24, axis=1).reshape(-1)
    cols = np.tile(edof, (1, 24)).reshape(-1)
    vals = (r[:, None, None] * k0[None, :, :]).reshape(-1)
    key = rows * n_dofs + cols
    uniq, inv = np.unique(key, return_inverse=True)
    acc = np.zeros(uniq.size)
    np.add.at(acc, inv, vals)
    urow, ucol = uniq // n_dofs, uniq % n_dofs
    row_ptr = np.zeros(n_dofs + 1, dtype=np.int64)
    np.add.at(row_ptr, urow + 1, 1)
    return np.cumsum(row_ptr), ucol.astype(np.int64), acc


def fem_matvec_assembled(nex, ney, nez, rho, K0, x):
    """y = K x through the assembled matrix (csr_spmv)."""
    rp, ci, v = fem_assemble(nex, ney, nez, rho, K0)
    return csr_spmv(rp, ci, v, x)


def fem_diagonal(nex, ney, nez, rho, K0):
    """The diagonal of the assembled K: every element adds rho_e K0[d, d] at
    each of its local dofs d."""
    edof = element_dofs(nex, ney, nez)
    n_dofs = 3 * (nex + 1) * (ney + 1) * (nez + 1)
    r = np.asarray(rho, dtype=np.float64)
    kd = np.diag(np.asarray(K0, dtype=np.float64))
    d = np.zeros(n_dofs)
    np.add.at(d, edof.reshape(-1), (r[:, None] * kd[None, :]).reshape(-1))
    return d
