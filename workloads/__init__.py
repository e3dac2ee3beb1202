"""Seeded synthetic sparse matrices and vectors shaped like the pages' workloads.

This module only draws inputs. It holds none of the method's arithmetic (no
product, no encoding), so both the oracle's tests and the library's tests and
benchmark can use it without sharing any of the computation under test.

Every generator uses ``numpy.random.Generator(PCG64(seed))`` and returns a
:class:`CSRInput` with int32 ``row_ptr``/``col_idx``, typed ``values`` and the
vector ``x``. Columns are strictly increasing inside each row.

Workloads (sizes and value distributions as the pages describe them):

* ``tiny``       -- 1000 x 1000, exactly 5 distinct random columns per row,
  fp32 values and x from U(-1, 1).
* ``laplacian``  -- 2-D 5-point Laplacian on an nx x ny grid (row r = i + nx*j;
  diagonal 4, -1 for each existing N/S/E/W neighbour), fp32, x U(-1, 1).
  The SuiteSparse ``ecology2`` matrix that the "CUDA CSR SpMV optimisation"
  page (section 2.1) measures on has this 5-point shape at ~1M rows; this
  generator stands in for it.
* ``powerlaw``   -- web-graph shaped rows: Zipf(2.0) lengths clipped to
  [1, max_len] and rescaled to an exact total, random distinct columns, fp32
  values and x from U(0, 1). Stands in for ``web-Google`` (916,428 rows,
  5,105,039 nonzeros, longest row 4,334) from the SpGEMM page's table.
* ``llm``        -- a pruned fp16 weight matrix: Bernoulli(1 - sparsity) mask,
  values N(0, 0.02) with exact zeros redrawn, x fp16 N(0, 1). Stands in for the
  12288 x 12288 matrices of the MACKO-SpMV page, section 3.1.
* ``fem``        -- assembled stiffness pattern of a structured hexahedral mesh
  (8-node elements, 3 dofs per node) from random SPD 24 x 24 element matrices
  scaled by a density rho ~ U(0.001, 1), as in the topology-optimisation page.
* ``fem_simp``   -- inputs of the matrix-free operator on the same mesh: one
  SPD 24 x 24 element matrix K0 scaled per element by rho ~ U(0.001, 1) (the
  page's SIMP setting, in which all elements share one stiffness matrix up to
  the density factor), and x from U(-1, 1); returned as :class:`FemMesh`.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class CSRInput:
    name: str
    n_rows: int
    n_cols: int
    row_ptr: np.ndarray   # int32[n_rows + 1]
    col_idx: np.ndarray   # int32[nnz]
    values: np.ndarray    # float32 or float16 [nnz]
    x: np.ndarray         # same dtype as values, [n_cols]
    meta: dict = field(default_factory=dict)

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    @property
    def dtype(self):
        return self.values.dtype

    def row_lengths(self) -> np.ndarray:
        return np.diff(self.row_ptr.astype(np.int64))


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _row_ptr_from_lengths(lengths: np.ndarray) -> np.ndarray:
    rp = np.zeros(lengths.shape[0] + 1, dtype=np.int64)
    np.cumsum(lengths, out=rp[1:])
    if rp[-1] > np.iinfo(np.int32).max:
        raise ValueError("nonzero count does not fit int32 row pointers")
    return rp.astype(np.int32)


def distinct_sorted_columns(rng: np.random.Generator, lengths: np.ndarray,
                            n_cols: int) -> np.ndarray:
    """For each row i draw lengths[i] distinct columns uniformly from
    [0, n_cols) and return them sorted inside each row (int32, row-major).

    Duplicates inside a row are redrawn until none is left."""
    lengths = np.asarray(lengths, dtype=np.int64)
    if lengths.size and lengths.max() > n_cols:
        raise ValueError("a row is longer than the number of columns")
    n_rows = lengths.shape[0]
    total = int(lengths.sum())
    row_of = np.repeat(np.arange(n_rows, dtype=np.int64), lengths)
    base = row_of * np.int64(n_cols)
    cols = rng.integers(0, n_cols, size=total, dtype=np.int64)
    while True:
        key = base + cols
        key.sort(kind="stable")
        cols = key - base
        dup = np.nonzero(key[1:] == key[:-1])[0] + 1
        if dup.size == 0:
            break
        cols[dup] = rng.integers(0, n_cols, size=dup.size, dtype=np.int64)
    return cols.astype(np.int32)


def from_lengths(name: str, lengths, n_cols: int, seed: int,
                 dtype=np.float32, low: float = -1.0, high: float = 1.0,
                 x_low: float = -1.0, x_high: float = 1.0) -> CSRInput:
    """Random matrix with the given row lengths, distinct sorted columns,
    values U(low, high) and x U(x_low, x_high) in ``dtype``."""
    rng = _rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    cols = distinct_sorted_columns(rng, lengths, n_cols)
    vals = rng.uniform(low, high, size=cols.shape[0]).astype(dtype)
    x = rng.uniform(x_low, x_high, size=n_cols).astype(dtype)
    return CSRInput(name, int(lengths.shape[0]), int(n_cols),
                    _row_ptr_from_lengths(lengths), cols, vals, x,
                    {"seed": seed})


def tiny(seed: int = 1, n: int = 1000, per_row: int = 5) -> CSRInput:
    """n x n, exactly ``per_row`` distinct uniform columns per row."""
    lengths = np.full(n, per_row, dtype=np.int64)
    m = from_lengths("tiny", lengths, n, seed)
    m.meta.update({"n": n, "per_row": per_row})
    return m


def laplacian(nx: int = 1000, ny: int = 999, seed: int = 2) -> CSRInput:
    """5-point Laplacian on an nx x ny grid; row r = i + nx*j; columns sorted
    (S, W, centre, E, N); diagonal 4, -1 per existing neighbour."""
    n = nx * ny
    r = np.arange(n, dtype=np.int64)
    i = r % nx
    j = r // nx
    # candidate columns in increasing order and their existence masks
    cand = np.stack([r - nx, r - 1, r, r + 1, r + nx], axis=1)
    ok = np.stack([j > 0, i > 0, np.ones(n, bool), i < nx - 1, j < ny - 1],
                  axis=1)
    vals = np.where(np.arange(5) == 2, 4.0, -1.0)[None, :].repeat(n, axis=0)
    lengths = ok.sum(axis=1)
    cols = cand[ok].astype(np.int32)
    v = vals[ok].astype(np.float32)
    x = _rng(seed).uniform(-1.0, 1.0, size=n).astype(np.float32)
    return CSRInput("laplacian", n, n, _row_ptr_from_lengths(lengths), cols, v,
                    x, {"nx": nx, "ny": ny, "seed": seed})


def powerlaw_lengths(rng: np.random.Generator, n: int, nnz: int,
                     max_len: int, a: float = 2.0) -> np.ndarray:
    """Zipf(a) row lengths clipped to [1, max_len], rescaled so that they sum
    to exactly ``nnz``: L <- clip(floor(s*L + u), 1, max_len) with
    s = nnz / sum(L) and u ~ U(0, 1), then +-1 on randomly chosen eligible rows
    until the total is exact."""
    lengths = np.minimum(rng.zipf(a, size=n).astype(np.int64), max_len)
    scale = nnz / float(lengths.sum())
    u = rng.random(n)
    lengths = np.clip(np.floor(scale * lengths + u), 1, max_len).astype(np.int64)
    diff = nnz - int(lengths.sum())
    while diff != 0:
        if diff > 0:
            elig = np.nonzero(lengths < max_len)[0]
            pick = rng.choice(elig, size=min(diff, elig.size), replace=False)
            lengths[pick] += 1
        else:
            elig = np.nonzero(lengths > 1)[0]
            pick = rng.choice(elig, size=min(-diff, elig.size), replace=False)
            lengths[pick] -= 1
        diff = nnz - int(lengths.sum())
    return lengths


def powerlaw(n: int = 916_428, nnz: int = 5_105_039, max_len: int = 4_334,
             a: float = 2.0, seed: int = 3) -> CSRInput:
    """Web-graph shaped matrix (load-imbalance case)."""
    rng = _rng(seed)
    lengths = powerlaw_lengths(rng, n, nnz, max_len, a)
    cols = distinct_sorted_columns(rng, lengths, n)
    vals = rng.random(cols.shape[0]).astype(np.float32)
    x = rng.random(n).astype(np.float32)
    return CSRInput("powerlaw", n, n, _row_ptr_from_lengths(lengths), cols,
                    vals, x, {"n": n, "nnz": nnz, "max_len": max_len, "a": a,
                              "seed": seed})


def llm_seed(sparsity: float) -> int:
    return 40 + int(round(sparsity * 10))


def llm(sparsity: float, n: int = 12_288, seed: int | None = None,
        block_rows: int = 512) -> CSRInput:
    """Pruned fp16 weight: keep each entry with probability 1 - sparsity,
    values N(0, 0.02) in fp16 with exact zeros redrawn, x fp16 N(0, 1)."""
    if seed is None:
        seed = llm_seed(sparsity)
    rng = _rng(seed)
    keep_p = 1.0 - sparsity
    lengths = np.empty(n, dtype=np.int64)
    col_parts = []
    for r0 in range(0, n, block_rows):
        r1 = min(n, r0 + block_rows)
        keep = rng.random((r1 - r0, n)) < keep_p
        lengths[r0:r1] = keep.sum(axis=1)
        col_parts.append(np.nonzero(keep)[1].astype(np.int32))
    cols = (np.concatenate(col_parts) if col_parts
            else np.zeros(0, dtype=np.int32))
    vals = rng.normal(0.0, 0.02, size=cols.shape[0]).astype(np.float16)
    while True:
        z = np.nonzero(vals == 0)[0]   # catches +0.0 and -0.0
        if z.size == 0:
            break
        vals[z] = rng.normal(0.0, 0.02, size=z.size).astype(np.float16)
    x = rng.standard_normal(n).astype(np.float16)
    return CSRInput(f"llm{int(round(sparsity * 100))}", n, n,
                    _row_ptr_from_lengths(lengths), cols, vals, x,
                    {"n": n, "sparsity": sparsity, "seed": seed})


# local node offsets of an 8-node hexahedron (fixed order)
HEX_NODES = np.array([(0, 0, 0), (1, 0, 0), (1, 1, 0), (0, 1, 0),
                      (0, 0, 1), (1, 0, 1), (1, 1, 1), (0, 1, 1)],
                     dtype=np.int64)


def fem_element_matrices(rng: np.random.Generator, n_elem: int,
                         batch: int = 8192) -> np.ndarray:
    """Ke = rho_e * (sym(G G^T) / 24 + I) with G iid N(0, 1) 24 x 24 and
    rho_e ~ U(0.001, 1); sym(M) = (M + M^T) / 2 makes Ke exactly symmetric.
    Draw order: all rho first, then G element by element."""
    rho = rng.uniform(0.001, 1.0, size=n_elem)
    ke = np.empty((n_elem, 24, 24), dtype=np.float64)
    eye = np.eye(24)
    for e0 in range(0, n_elem, batch):
        e1 = min(n_elem, e0 + batch)
        g = rng.standard_normal((e1 - e0, 24, 24))
        m = g @ g.transpose(0, 2, 1)
        s = (m + m.transpose(0, 2, 1)) * 0.5
        ke[e0:e1] = rho[e0:e1, None, None] * (s / 24.0 + eye)
    return ke


def fem(nex: int = 120, ney: int = 60, nez: int = 30, seed: int = 5) -> CSRInput:
    """Assembled 3-D stiffness pattern: hex mesh nex x ney x nez, element
    e = ex + nex*(ey + ney*ez), node = i + nnx*(j + nny*k), dof = 3*node + c.
    Assembly is a fp64 sum over elements in element order, rounded to fp32
    once; every node pair that shares an element is a stored entry."""
    rng = _rng(seed)
    nnx, nny, nnz_ = nex + 1, ney + 1, nez + 1
    n_nodes = nnx * nny * nnz_
    n = 3 * n_nodes
    n_elem = nex * ney * nez
    ke = fem_element_matrices(rng, n_elem)

    e = np.arange(n_elem, dtype=np.int64)
    ex, ey, ez = e % nex, (e // nex) % ney, e // (nex * ney)
    node = ((ex[:, None] + HEX_NODES[None, :, 0])
            + nnx * ((ey[:, None] + HEX_NODES[None, :, 1])
                     + nny * (ez[:, None] + HEX_NODES[None, :, 2])))  # [E, 8]
    # neighbour slot of local node b seen from local node a: offsets in
    # {-1,0,1}^3 ordered by (dz, dy, dx) so that slot order = column order
    d = HEX_NODES[None, :, :] - HEX_NODES[:, None, :]              # [8, 8, 3]
    nb = (d[..., 2] + 1) * 9 + (d[..., 1] + 1) * 3 + (d[..., 0] + 1)  # [8, 8]
    alpha = np.arange(24)
    a_of, c_of = alpha // 3, alpha % 3
    local_slot = nb[a_of[:, None], a_of[None, :]] * 3 + c_of[None, :]  # [24,24]
    row_dof = 3 * node[:, a_of] + c_of[None, :]                     # [E, 24]
    bins = row_dof[:, :, None] * 81 + local_slot[None, :, :]        # [E,24,24]
    acc = np.bincount(bins.reshape(-1), weights=ke.reshape(-1),
                      minlength=n * 81)
    del bins, ke

    # which of the 27 neighbour nodes exist, per node
    nid = np.arange(n_nodes, dtype=np.int64)
    ni, nj, nk = nid % nnx, (nid // nnx) % nny, nid // (nnx * nny)
    off = np.array([(dx, dy, dz) for dz in (-1, 0, 1) for dy in (-1, 0, 1)
                    for dx in (-1, 0, 1)], dtype=np.int64)          # [27, 3]
    ii = ni[:, None] + off[None, :, 0]
    jj = nj[:, None] + off[None, :, 1]
    kk = nk[:, None] + off[None, :, 2]
    exists = ((ii >= 0) & (ii < nnx) & (jj >= 0) & (jj < nny)
              & (kk >= 0) & (kk < nnz_))                             # [N, 27]
    nb_node = ii + nnx * (jj + nny * kk)
    valid = np.repeat(np.repeat(exists, 3, axis=1), 3, axis=0)      # [n, 81]
    col = 3 * np.repeat(np.repeat(nb_node, 3, axis=1), 3, axis=0) \
        + np.tile(np.arange(3), 27)[None, :]
    lengths = valid.sum(axis=1)
    cols = col[valid].astype(np.int32)
    vals = acc.reshape(n, 81)[valid].astype(np.float32)
    x = rng.uniform(-1.0, 1.0, size=n).astype(np.float32)
    return CSRInput("fem", n, n, _row_ptr_from_lengths(lengths), cols, vals, x,
                    {"nex": nex, "ney": ney, "nez": nez, "seed": seed})


def fem_nnz(nex: int, ney: int, nez: int) -> int:
    """Closed-form stored-entry count of the assembled hex pattern: 9 times
    the product over axes of (3 m - 2), m = nodes along the axis."""
    return 9 * (3 * (nex + 1) - 2) * (3 * (ney + 1) - 2) * (3 * (nez + 1) - 2)


@dataclass
class FemMesh:
    """Inputs of the matrix-free stiffness operator on a structured hex mesh:
    element e = ex + nex*(ey + ney*ez) has matrix rho[e] * K0; nodes, dofs
    and the local node order are those of ``fem`` (HEX_NODES)."""
    name: str
    nex: int
    ney: int
    nez: int
    rho: np.ndarray      # float32[n_elem]
    K0: np.ndarray       # float32[24, 24], symmetric positive definite
    x: np.ndarray        # float32[n_dofs]
    params: dict = field(default_factory=dict)

    @property
    def n_elem(self) -> int:
        return self.nex * self.ney * self.nez

    @property
    def n_nodes(self) -> int:
        return (self.nex + 1) * (self.ney + 1) * (self.nez + 1)

    @property
    def n_dofs(self) -> int:
        return 3 * self.n_nodes


def fem_simp(nex: int = 120, ney: int = 60, nez: int = 30, seed: int = 6) -> FemMesh:
    """Densities rho_e ~ U(0.001, 1) scaling one element matrix
    K0 = sym(G G^T) / 24 + I (G iid N(0, 1), computed in fp64 and rounded to
    fp32 once, so K0 stays exactly symmetric), and x ~ U(-1, 1). Draw order:
    rho, G, x."""
    rng = _rng(seed)
    n_elem = nex * ney * nez
    rho = rng.uniform(0.001, 1.0, size=n_elem).astype(np.float32)
    g = rng.standard_normal((24, 24))
    m = g @ g.T
    k0 = ((m + m.T) * 0.5 / 24.0 + np.eye(24)).astype(np.float32)
    n_dofs = 3 * (nex + 1) * (ney + 1) * (nez + 1)
    x = rng.uniform(-1.0, 1.0, size=n_dofs).astype(np.float32)
    return FemMesh(f"fem_simp_{nex}x{ney}x{nez}", nex, ney, nez, rho, k0, x,
                   {"seed": seed})


WORKLOADS = {
    "tiny": lambda: tiny(),
    "laplacian": lambda: laplacian(),
    "powerlaw": lambda: powerlaw(),
    "llm30": lambda: llm(0.3),
    "llm50": lambda: llm(0.5),
    "llm70": lambda: llm(0.7),
    "llm90": lambda: llm(0.9),
    "fem": lambda: fem(),
}


def make(name: str) -> CSRInput:
    """Full-size workload by name (see WORKLOADS)."""
    return WORKLOADS[name]()
