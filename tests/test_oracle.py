"""Pins for the oracle: each check compares it with something other than
itself (a pure-Python dense product, a closed form, scipy, the page's worked
example, hand-derived encodings, invariants). The last test plants mistakes
in copies of the oracle's C source and checks that some pin fails for each.
"""
import json
import os
import sys

import numpy as np
import pytest
import scipy.sparse as sp

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "delta_examples.json")
GOLDEN_WIDTHS = os.path.join(os.path.dirname(__file__), "golden", "delta_widths.json")


# ---------------------------------------------------------------- helpers

def random_csr(seed, n_rows, n_cols, density=0.3, dtype=np.float32,
               empty_rows=(), full_rows=()):
    rng = np.random.default_rng(seed)
    mask = rng.random((n_rows, n_cols)) < density
    for r in empty_rows:
        mask[r] = False
    for r in full_rows:
        mask[r] = True
    rows, cols = np.nonzero(mask)
    lengths = mask.sum(axis=1)
    rp = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    vals = rng.uniform(-1, 1, size=rows.size).astype(dtype)
    x = rng.uniform(-1, 1, size=n_cols).astype(dtype)
    return rp, cols.astype(np.int32), vals, x


def dense_rows(rp, ci, vals, n_cols):
    """Dense matrix as Python lists of floats (fp64)."""
    n_rows = len(rp) - 1
    a = [[0.0] * n_cols for _ in range(n_rows)]
    for i in range(n_rows):
        for k in range(int(rp[i]), int(rp[i + 1])):
            a[i][int(ci[k])] = float(vals[k])
    return a


def dense_matvec(a, x):
    """Textbook dense product, column order, pure Python."""
    y, s = [], []
    for row in a:
        acc = 0.0
        acc_abs = 0.0
        for j, aij in enumerate(row):
            p = aij * float(x[j])
            acc = acc + p
            acc_abs = acc_abs + abs(p)
        y.append(acc)
        s.append(acc_abs)
    return np.array(y), np.array(s)


# ---------------------------------------------------------------- pins

def pin_dense_bruteforce():
    cases = [
        dict(seed=11, n_rows=17, n_cols=23, density=0.3),
        dict(seed=12, n_rows=40, n_cols=9, density=0.5, empty_rows=(0, 5, 39)),
        dict(seed=13, n_rows=32, n_cols=64, density=0.1, full_rows=(3, 31)),
        dict(seed=14, n_rows=1, n_cols=1, density=1.0),
        dict(seed=15, n_rows=64, n_cols=64, density=0.05, dtype=np.float16),
    ]
    for c in cases:
        rp, ci, vals, x = random_csr(**c)
        y, s = oracle.csr_spmv(rp, ci, vals, x)
        y_ref, s_ref = dense_matvec(dense_rows(rp, ci, vals, c["n_cols"]), x)
        # zeros add exactly and columns are sorted: bit-for-bit equal
        assert np.array_equal(y, y_ref), c
        assert np.array_equal(s, s_ref), c


def pin_identity_and_permutation():
    rng = np.random.default_rng(21)
    n = 257
    x = rng.uniform(-1, 1, n).astype(np.float32)
    rp = np.arange(n + 1, dtype=np.int32)
    eye_cols = np.arange(n, dtype=np.int32)
    ones = np.ones(n, dtype=np.float32)
    y, s = oracle.csr_spmv(rp, eye_cols, ones, x)
    assert np.array_equal(y, x.astype(np.float64))
    assert np.array_equal(s, np.abs(x).astype(np.float64))
    perm = rng.permutation(n).astype(np.int32)
    y = oracle.csr_spmv(rp, perm, ones, x, with_abs=False)
    assert np.array_equal(y, x[perm].astype(np.float64))
    # a non-symmetric permutation distinguishes P x from P^T x
    inv = np.argsort(perm)
    assert not np.array_equal(x[perm], x[inv])


def pin_laplacian_constant():
    nx, ny = 9, 7
    m = workloads.laplacian(nx, ny, seed=0)
    nbrs = m.row_lengths() - 1
    r = np.arange(m.n_rows)
    interior = (r % nx > 0) & (r % nx < nx - 1) & (r // nx > 0) & (r // nx < ny - 1)
    # any finite c: the sorted-order partial sums are -c, -2c, 2c, c, 0
    for c in (0.7318937, -3.25e7, 1.0e-30):
        y = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values,
                            np.full(m.n_rows, c, np.float64), with_abs=False)
        assert np.all(y[interior] == 0.0)
    # boundary rows: c * (4 - #neighbours); dyadic c keeps every partial exact
    for c in (0.75, -1.5, 2.0 ** -10 * 3):
        y = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values,
                            np.full(m.n_rows, c, np.float64), with_abs=False)
        assert np.array_equal(y, c * (4.0 - nbrs))


def pin_row_of_ones():
    rng = np.random.default_rng(31)
    n = 1000
    x = rng.uniform(-1, 1, n)
    rp = np.array([0, n], dtype=np.int32)
    y, s = oracle.csr_spmv(rp, np.arange(n, dtype=np.int32),
                           np.ones(n, np.float32), x)
    acc = 0.0
    acc_abs = 0.0
    for v in x:
        acc = acc + float(v)
        acc_abs = acc_abs + abs(float(v))
    assert y[0] == acc and s[0] == acc_abs


def pin_scipy():
    mats = [workloads.tiny(), workloads.laplacian(40, 30),
            workloads.powerlaw(n=5000, nnz=27000, max_len=300),
            workloads.fem(4, 3, 2), workloads.llm(0.7, n=256)]
    for m in mats:
        y, s = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, m.x)
        a = sp.csr_matrix((m.values.astype(np.float64), m.col_idx, m.row_ptr),
                          shape=(m.n_rows, m.n_cols))
        y_sp = a @ m.x.astype(np.float64)
        assert np.all(np.abs(y - y_sp) <= 1e-14 * s + 1e-300), m.name
        s_sp = abs(a) @ np.abs(m.x.astype(np.float64))
        assert np.allclose(s, s_sp, rtol=1e-13, atol=0), m.name


def pin_delta_golden():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        cols = np.array(c["cols"], dtype=np.int64)
        n = cols.size
        vals = (np.arange(1, n + 1) * 0.125).astype(np.float16)
        rp = np.array([0, n], dtype=np.int64)
        m = oracle.delta_encode(64, rp, cols, vals)
        d = m.deltas()
        if c["kind"] == "printed":
            kept = m.values != 0
            assert list(d[kept][:len(c["deltas_prefix"])]) == c["deltas_prefix"]
            continue
        assert list(d) == c["deltas"], c
        assert list((m.values == 0).astype(int)) == c["pad"], c
        assert list(m.words) == c["words"], c
        assert m.n_entries % 8 == 0
        # non-padding entries carry the input values in order
        assert np.array_equal(m.values[m.values != 0], vals.view(np.uint16))


def pin_delta_widths_golden():
    with open(GOLDEN_WIDTHS) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        bits = c["bits"]
        cols = np.array(c["cols"], dtype=np.int64)
        n = cols.size
        vals = (np.arange(1, n + 1) * 0.125).astype(np.float16)
        rp = np.array([0, n], dtype=np.int64)
        m = oracle.delta_encode(512, rp, cols, vals, bits=bits)
        assert list(m.deltas()) == c["deltas"], c
        assert list((m.values == 0).astype(int)) == c["pad"], c
        assert list(m.words) == c["words"], c
        assert m.n_entries % (32 // bits) == 0
        assert np.array_equal(m.values[m.values != 0], vals.view(np.uint16))


def expected_pad_counts(rp, ci, bits=4):
    """Closed form of the reading: with b-bit fields a gap d (first gap =
    first column) needs max(0, floor((d - 1) / (2^b - 1))) padding entries
    (floor((d - 1) / 15) for 4 bits); rows round up to 32 / b entries."""
    rp = np.asarray(rp, np.int64)
    ci = np.asarray(ci, np.int64)
    n_rows = rp.size - 1
    lengths = np.diff(rp)
    prev = np.zeros_like(ci)
    first = np.zeros(ci.size, bool)
    first[rp[:-1][lengths > 0]] = True
    prev[~first] = ci[np.nonzero(~first)[0] - 1]
    gaps = ci - prev
    dmax = (1 << bits) - 1
    per = 32 // bits
    pads_per = np.maximum(0, (gaps - 1) // dmax)
    row_of = np.repeat(np.arange(n_rows), lengths)
    row_pads = np.bincount(row_of, weights=pads_per, minlength=n_rows).astype(np.int64)
    unaligned = lengths + row_pads
    aligned = (unaligned + per - 1) // per * per
    return int(pads_per.sum()), int((aligned - unaligned).sum()), aligned


def pin_delta_roundtrip_and_counts():
    mats = [workloads.llm(0.3, n=200), workloads.llm(0.9, n=333),
            workloads.from_lengths("mixed", np.r_[0, 1, 7, 8, 9, 0, 64, 3],
                                   400, seed=5, dtype=np.float16)]
    for m, bits in [(mm, b) for mm in mats for b in (4, 2, 8)]:
        vals = m.values.astype(np.float16)
        vals[vals == 0] = np.float16(0.5)   # the round trip needs no +-0.0
        enc = oracle.delta_encode(m.n_cols, m.row_ptr, m.col_idx, vals, bits=bits)
        gaps, aligns, aligned = expected_pad_counts(m.row_ptr, m.col_idx, bits)
        assert enc.gap_pads == gaps and enc.align_pads == aligns
        assert np.array_equal(np.diff(enc.row_ptr), aligned)
        assert enc.n_entries == m.nnz + gaps + aligns
        d = enc.deltas()
        assert d.max(initial=0) <= (1 << bits) - 1
        rp, col, v = oracle.delta_decode(enc)
        assert np.array_equal(rp, m.row_ptr.astype(np.int64))
        assert np.array_equal(col, m.col_idx.astype(np.int64))
        assert np.array_equal(v.view(np.uint16), vals.view(np.uint16))
        # columns rebuilt by a running sum of the codes, row by row
        for r in range(min(m.n_rows, 20)):
            e0, e1 = enc.row_ptr[r], enc.row_ptr[r + 1]
            c = np.cumsum(d[e0:e1].astype(np.int64))
            kept = enc.values[e0:e1] != 0
            assert np.array_equal(c[kept], m.col_idx[m.row_ptr[r]:m.row_ptr[r + 1]])


GOLDEN_SELL = os.path.join(os.path.dirname(__file__), "golden", "sell_examples.json")


def pin_sell_golden():
    """Hand-worked sliced-ELL layouts (row order, length-sorted windows,
    plain ELL as one slice) and the CV bands, boundaries included."""
    from oracle import sell
    g = json.load(open(GOLDEN_SELL))
    mt = g["matrix"]
    rp = np.array(mt["row_ptr"], np.int64)
    ci = np.array(mt["col_idx"], np.int32)
    vals = np.array(mt["values"], np.float32)
    for lay in g["layouts"]:
        m = sell.sell_encode(mt["n_cols"], rp, ci, vals, C=lay["C"], sigma=lay["sigma"])
        assert m.slice_ptr.tolist() == lay["slice_ptr"], lay
        assert m.perm.tolist() == lay["perm"], lay
        assert m.cols.tolist() == lay["cols"], lay
        assert m.vals.tolist() == lay["vals"], lay
    for case in g["cv_cases"]:
        rp2 = np.concatenate([[0], np.cumsum(case["lengths"])])
        assert abs(sell.row_length_cv(rp2) - case["cv"]) <= 1e-12 * max(1.0, case["cv"])
        assert list(sell.select_format(rp2)) == case["choice"], case


def pin_sell_invariants():
    """On random matrices (empty rows, ties, a ragged last slice): every row's
    slots hold its entries in order and then value-0 padding at in-range
    columns; slice widths are the slices' longest rows; perm is a permutation
    whose windows are sorted by decreasing length, ties in row order; and
    the product read from the layout equals the CSR product exactly."""
    from oracle import sell
    rng = np.random.default_rng(31)
    for n, n_cols, C, sigma in ((101, 50, 32, 1), (101, 50, 32, 16), (77, 9, 7, 1000),
                                (64, 200, 32, 64), (5, 3, 32, 1), (0, 4, 32, 1)):
        lengths = rng.integers(0, min(n_cols, 12) + 1, n)
        lengths[::9] = 0
        rp = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
        ci = np.concatenate([np.sort(rng.choice(n_cols, L, replace=False)) for L in lengths]
                            ).astype(np.int32) if n else np.zeros(0, np.int32)
        vals = rng.uniform(0.5, 1.5, rp[-1]).astype(np.float32)
        m = sell.sell_encode(n_cols, rp, ci, vals, C=C, sigma=sigma)
        perm = m.perm[:n]
        assert sorted(perm.tolist()) == list(range(n)) and np.all(m.perm[n:] == -1)
        for w0 in range(0, n, max(sigma, 1)):
            win = perm[w0:w0 + max(sigma, 1)]
            L = lengths[win]
            assert np.all(L[:-1] >= L[1:])
            for a, b in zip(win[:-1], win[1:]):
                if lengths[a] == lengths[b]:
                    assert a < b
        for sl in range(m.n_slices):
            w = (m.slice_ptr[sl + 1] - m.slice_ptr[sl]) // C
            rows = [r for r in m.perm[sl * C:(sl + 1) * C] if r >= 0]
            assert w == max([lengths[r] for r in rows], default=0)
            for lane in range(C):
                r = m.perm[sl * C + lane]
                at = m.slice_ptr[sl] + np.arange(w) * C + lane
                if r < 0:
                    assert np.all(m.vals[at] == 0) and np.all(m.cols[at] == 0)
                    continue
                L = lengths[r]
                assert np.array_equal(m.cols[at[:L]], ci[rp[r]:rp[r + 1]])
                assert np.array_equal(m.vals[at[:L]], vals[rp[r]:rp[r + 1]])
                assert np.all(m.vals[at[L:]] == 0)
                assert np.all(m.cols[at[L:]] == (ci[rp[r + 1] - 1] if L else 0))
        assert sell.sell_slot_count(rp, C, sigma) == (m.n_slots, m.n_slices)
        x = rng.uniform(-1, 1, n_cols)
        y1, s1 = sell.sell_spmv(m, x)
        y2, s2 = oracle.csr_spmv(rp, ci, vals, x)
        assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


def pin_fem_single_element():
    """One element: the hand-derived dof table (corners in the order
    (0,0,0) (1,0,0) (1,1,0) (0,1,0) then the top face; node = i + 2 j + 4 k),
    and a K0 with one nonzero entry K0[a, b] = 1 moves rho * x[dof b] to
    dof a and nothing else (a transposed K0 or a wrong dof fails)."""
    from oracle import fem
    edof = fem.element_dofs(1, 1, 1)
    assert edof.tolist() == [[0, 1, 2, 3, 4, 5, 9, 10, 11, 6, 7, 8, 12, 13, 14,
                              15, 16, 17, 21, 22, 23, 18, 19, 20]]
    x = np.arange(1, 25, dtype=np.float64) * 0.5
    for a, b in ((0, 0), (2, 17), (23, 5), (7, 20)):
        k0 = np.zeros((24, 24))
        k0[a, b] = 1.0
        y, s = fem.fem_matvec(1, 1, 1, [2.0], k0, x)
        want = np.zeros(24)
        want[edof[0, a]] = 2.0 * x[edof[0, b]]
        assert np.array_equal(y, want) and np.array_equal(s, np.abs(want))


def pin_fem_identity_closed_form():
    """K0 = I, rho = 1: y at a dof is x times the number of elements around
    its node, the product over the axes of 1 (mesh boundary) or 2 (inside)."""
    from oracle import fem
    nex, ney, nez = 4, 3, 2
    # eighths: every partial sum of up to 8 copies is exact
    x = np.random.default_rng(3).integers(-64, 65, 3 * 5 * 4 * 3) / 8.0
    y, _ = fem.fem_matvec(nex, ney, nez, np.ones(nex * ney * nez), np.eye(24), x)
    mult = np.zeros(5 * 4 * 3)
    for k in range(3):
        for j in range(4):
            for i in range(5):
                m = ((1 if i in (0, nex) else 2) * (1 if j in (0, ney) else 2)
                     * (1 if k in (0, nez) else 2))
                mult[i + 5 * (j + 4 * k)] = m
    assert np.array_equal(y, np.repeat(mult, 3) * x)


def pin_fem_assembled_routes():
    """The element loop equals the assembled matrix's product; the assembled
    pattern is the one the fem workload generator builds independently, its
    size is the closed form, and K is symmetric positive definite."""
    from oracle import fem
    m = workloads.fem_simp(5, 4, 3, seed=9)
    y, s = fem.fem_matvec(m.nex, m.ney, m.nez, m.rho, m.K0, m.x)
    y2, s2 = fem.fem_matvec_assembled(m.nex, m.ney, m.nez, m.rho, m.K0, m.x)
    assert np.all(np.abs(y - y2) <= 1e-13 * s)
    assert np.all(s2 <= s * (1 + 1e-12))
    rp, ci, v = fem.fem_assemble(m.nex, m.ney, m.nez, m.rho, m.K0)
    ref = workloads.fem(5, 4, 3)
    assert np.array_equal(rp, ref.row_ptr) and np.array_equal(ci, ref.col_idx)
    assert rp[-1] == workloads.fem_nnz(5, 4, 3)
    A = sp.csr_matrix((v, ci, rp), shape=(m.n_dofs, m.n_dofs))
    assert abs(A - A.T).max() == 0
    assert np.allclose(fem.fem_diagonal(m.nex, m.ney, m.nez, m.rho, m.K0), A.diagonal(),
                       rtol=1e-15, atol=0)
    rng = np.random.default_rng(1)
    for _ in range(3):
        z = rng.standard_normal(m.n_dofs)
        assert z @ (A @ z) > 0


def pin_pcg_closed_forms():
    """Jacobi-PCG: on a diagonal matrix the preconditioner is the inverse,
    so one step lands on b / d exactly; on 2 x 2 [[4, 1], [1, 3]] x = [1, 2]
    two steps give the exact [1/11, 7/11] (CG ends in n steps); on a random
    SPD 40 x 40 system it reaches the direct solution within n + 2 steps;
    an indefinite matrix breaks down (p . A p = 0) and a step limit stops."""
    from oracle import pcg
    d = np.array([2.0, 4.0, 0.5, 8.0])
    b = np.array([1.0, -2.0, 3.0, 0.25])
    x, it, st, _ = pcg.jacobi_pcg(lambda v: d * v, d, b, np.zeros(4), 1e-12, 50)
    assert it == 1 and st == 1 and np.array_equal(x, b / d)
    A = np.array([[4.0, 1.0], [1.0, 3.0]])
    x, it, st, _ = pcg.jacobi_pcg(lambda v: A @ v, np.diag(A), np.array([1.0, 2.0]),
                                  np.zeros(2), 1e-14, 2)
    assert it <= 2 and np.allclose(x, [1 / 11, 7 / 11], rtol=0, atol=1e-15)
    rng = np.random.default_rng(5)
    G = rng.standard_normal((40, 40))
    A = G @ G.T + 40 * np.eye(40)
    b = rng.standard_normal(40)
    x, it, st, hist = pcg.jacobi_pcg(lambda v: A @ v, np.diag(A), b, np.zeros(40), 1e-12, 42)
    assert st == 1 and it <= 42
    assert np.allclose(x, np.linalg.solve(A, b), rtol=0, atol=1e-9)
    D = np.diag([1.0, -1.0])
    x, it, st, _ = pcg.jacobi_pcg(lambda v: D @ v, np.diag(D), np.ones(2), np.zeros(2), 1e-12, 5)
    assert st == 3
    x, it, st, _ = pcg.jacobi_pcg(lambda v: A @ v, np.diag(A), b, np.zeros(40), 1e-14, 3)
    assert st == 2 and it == 3


ALL_PINS = [pin_dense_bruteforce, pin_identity_and_permutation,
            pin_laplacian_constant, pin_row_of_ones, pin_scipy,
            pin_delta_golden, pin_delta_widths_golden, pin_delta_roundtrip_and_counts,
            pin_sell_golden, pin_sell_invariants,
            pin_fem_single_element, pin_fem_identity_closed_form, pin_fem_assembled_routes,
            pin_pcg_closed_forms]


# ---------------------------------------------------------------- tests

@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_delta_rejects_unsorted_or_duplicate():
    rp = np.array([0, 3], np.int64)
    vals = np.ones(3, np.float16)
    with pytest.raises(ValueError):
        oracle.delta_encode(10, rp, np.array([1, 5, 3]), vals)
    with pytest.raises(ValueError):
        oracle.delta_encode(10, rp, np.array([1, 5, 5]), vals)


def test_delta_spmv_equals_csr_spmv():
    m = workloads.llm(0.5, n=300)
    enc = oracle.delta_encode(m.n_cols, m.row_ptr, m.col_idx, m.values)
    y1, s1 = oracle.delta_spmv(enc, m.x)
    y2, s2 = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, m.x)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


def test_all_core_baseline_equals_oracle():
    """The OpenMP baseline shares the rows out over threads but sums each row
    in the oracle's order, so its y is the oracle's bit for bit (CSR and the
    three delta widths)."""
    from oracle import parallel
    m = workloads.powerlaw(n=20000, nnz=111000, max_len=3000)
    y0 = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, m.x, with_abs=False)
    assert np.array_equal(y0, parallel.CsrOperands(m.row_ptr, m.col_idx, m.values, m.x)())
    w = workloads.llm(0.7, n=600)
    for bits in (2, 4, 8):
        enc = oracle.delta_encode(w.n_cols, w.row_ptr, w.col_idx, w.values, bits=bits)
        y1 = oracle.delta_spmv(enc, w.x, with_abs=False)
        assert np.array_equal(y1, parallel.DeltaOperands(enc, w.x)())
    assert parallel.threads() >= 1


# mutations of the oracle source: (name, old text, new text)
MUTANTS = [
    ("dropped_term", "k < row_ptr[i + 1]; ++k) {\n      double prod",
     "k < row_ptr[i + 1] - 1; ++k) {\n      double prod"),
    ("wrong_sign", "acc = acc + prod;", "acc = acc - prod;"),
    ("wrong_x_index", "values[k] * x[col_idx[k]]",
     "values[k] * x[col_idx[row_ptr[i]]]"),
    ("wrong_value_index", "values[k] * x[col_idx[k]]",
     "values[row_ptr[i]] * x[col_idx[k]]"),
    ("abs_sum_signed", "(prod < 0.0 ? -prod : prod)", "prod"),
    ("pad_threshold", "const int64_t dmax = ((int64_t)1 << bits) - 1; /* largest",
     "const int64_t dmax = ((int64_t)1 << bits) - 2; /* largest"),
    ("prev_not_reset", "int64_t prev = 0;", "int64_t prev = 1;"),
    ("nibble_order", "uint32_t shift = (uint32_t)(bits * (e % per_word));\n  out_words",
     "uint32_t shift = (uint32_t)(bits * (per_word - 1 - e % per_word));\n  out_words"),
    ("no_row_alignment", "count % per_word != 0", "count % 1 != 0"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = oracle.source_text()
    assert old in src, name
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path), name)
    failures = 0
    with oracle.use_library(lib):
        for pin in ALL_PINS:
            try:
                pin()
            except (AssertionError, ValueError, IndexError):
                failures += 1
    assert failures > 0, f"no pin caught mutant {name}"


# ---------------------------------------------------------------- generators

def test_tiny_shape():
    m = workloads.tiny()
    assert m.n_rows == 1000 and m.nnz == 5000
    assert np.all(m.row_lengths() == 5)
    for r in range(m.n_rows):
        c = m.col_idx[m.row_ptr[r]:m.row_ptr[r + 1]]
        assert np.all(np.diff(c) > 0)
    assert m.values.dtype == np.float32 and np.all(np.abs(m.values) <= 1)


def test_laplacian_counts():
    for nx, ny in ((1, 1), (1, 6), (5, 1), (13, 4)):
        m = workloads.laplacian(nx, ny)
        assert m.nnz == 5 * nx * ny - 2 * nx - 2 * ny
    m = workloads.laplacian()
    assert (m.n_rows, m.nnz) == (999_000, 4_991_002)


def test_powerlaw_stats():
    m = workloads.powerlaw()
    L = m.row_lengths()
    assert m.n_rows == 916_428 and m.nnz == 5_105_039
    assert L.min() >= 1 and L.max() <= 4334
    assert 0.55 < (L == 1).mean() < 0.75
    key = np.repeat(np.arange(m.n_rows, dtype=np.int64), L) * m.n_cols + m.col_idx
    assert np.all(np.diff(key) > 0)   # sorted, distinct inside rows


def test_fem_structure():
    assert workloads.fem_nnz(120, 60, 30) == 53_514_279
    m = workloads.fem(5, 4, 3)
    assert m.n_rows == 3 * 6 * 5 * 4
    assert m.nnz == workloads.fem_nnz(5, 4, 3)
    assert m.row_lengths().max() == 81
    a = sp.csr_matrix((m.values, m.col_idx, m.row_ptr), shape=(m.n_rows,) * 2)
    assert (a != a.T).nnz == 0          # bit-exact symmetry
    rng = np.random.default_rng(0)
    ad = a.astype(np.float64)
    for _ in range(5):
        v = rng.standard_normal(m.n_rows)
        assert v @ (ad @ v) > 0


def test_llm_values():
    m = workloads.llm(0.5, n=512)
    assert m.values.dtype == np.float16 and m.x.dtype == np.float16
    assert not np.any(m.values == 0)
    assert abs(m.nnz / 512 ** 2 - 0.5) < 0.01
    assert workloads.llm_seed(0.3) == 43 and workloads.llm_seed(0.9) == 49


SELL_MUTANTS = {
    "transposed_slots": ("at = slice_ptr[s] + k * C + lane", "at = slice_ptr[s] + lane * widths[s] + k"),
    "ascending_sort": ('np.argsort(-lengths[w0:w1], kind="stable")',
                       'np.argsort(lengths[w0:w1], kind="stable")'),
    "padding_at_column_0": ("cols[at[~real]] = ci[rp[i + 1] - 1]", "pass"),
    "sample_std": ("np.sqrt(np.mean((lengths - mean) ** 2))",
                   "np.sqrt(np.sum((lengths - mean) ** 2) / max(lengths.size - 1, 1))"),
    "strict_upper_band": ("if cv <= CV_CSR:", "if cv < CV_CSR:"),
}


@pytest.mark.parametrize("name", list(SELL_MUTANTS))
def test_sell_planted_mistake_is_caught(name):
    """A plausible mistake planted in the sliced-ELL oracle (on the CPU)
    fails one of its pins."""
    import types
    import oracle.sell as real
    old, new = SELL_MUTANTS[name]
    src = open(real.__file__).read()
    assert src.count(old) == 1
    mutant = types.ModuleType("oracle.sell")
    mutant.__package__ = "oracle"
    exec(compile(src.replace(old, new), real.__file__ + ":" + name, "exec"), mutant.__dict__)
    saved = sys.modules["oracle.sell"]
    sys.modules["oracle.sell"] = mutant
    oracle.sell = mutant
    try:
        failed = False
        for pin in (pin_sell_golden, pin_sell_invariants):
            try:
                pin()
            except AssertionError:
                failed = True
        assert failed, f"planted mistake {name} passed every pin"
    finally:
        sys.modules["oracle.sell"] = saved
        oracle.sell = saved


FEM_MUTANTS = {
    "corner_order": ("(1, 1, 0), (0, 1, 0),\n                    (0, 0, 1)",
                     "(0, 1, 0), (1, 1, 0),\n                    (0, 0, 1)"),
    "transposed_K0": ("f = r[:, None] * (u @ k0.T)", "f = r[:, None] * (u @ k0)"),
    "node_stride": ("node = i + (nex + 1) * (j + (ney + 1) * k)",
                    "node = i + nex * (j + ney * k)"),
    "dropped_density": ("f = r[:, None] * (u @ k0.T)", "f = (u @ k0.T)"),
}


@pytest.mark.parametrize("name", list(FEM_MUTANTS))
def test_fem_planted_mistake_is_caught(name):
    """A plausible mistake planted in the matrix-free oracle (on the CPU)
    fails one of its pins."""
    import types
    import oracle.fem as real
    old, new = FEM_MUTANTS[name]
    src = open(real.__file__).read()
    assert src.count(old) == 1, name
    mutant = types.ModuleType("oracle.fem")
    mutant.__package__ = "oracle"
    exec(compile(src.replace(old, new), real.__file__ + ":" + name, "exec"), mutant.__dict__)
    saved = sys.modules["oracle.fem"]
    sys.modules["oracle.fem"] = mutant
    oracle.fem = mutant
    try:
        failed = False
        for pin in (pin_fem_single_element, pin_fem_identity_closed_form,
                    pin_fem_assembled_routes):
            try:
                pin()
            except (AssertionError, IndexError, ValueError):
                failed = True
        assert failed, f"planted mistake {name} passed every pin"
    finally:
        sys.modules["oracle.fem"] = saved
        oracle.fem = saved


PCG_MUTANTS = {
    "no_preconditioner": ("z = dinv * r\n        rz_new", "z = r\n        rz_new"),
    "residual_sign": ("r -= alpha * q", "r += alpha * q"),
    "beta_inverted": ("beta = rz_new / rz", "beta = rz / rz_new"),
    "direction_without_z": ("p = z + beta * p", "p = r + beta * p"),
}


@pytest.mark.parametrize("name", list(PCG_MUTANTS))
def test_pcg_planted_mistake_is_caught(name):
    """A plausible mistake planted in the CG oracle (on the CPU) fails its
    pins."""
    import types
    import oracle.pcg as real
    old, new = PCG_MUTANTS[name]
    src = open(real.__file__).read()
    assert src.count(old) == 1, name
    mutant = types.ModuleType("oracle.pcg")
    mutant.__package__ = "oracle"
    exec(compile(src.replace(old, new), real.__file__ + ":" + name, "exec"), mutant.__dict__)
    saved = sys.modules["oracle.pcg"]
    sys.modules["oracle.pcg"] = mutant
    oracle.pcg = mutant
    try:
        with pytest.raises(AssertionError):
            pin_pcg_closed_forms()
    finally:
        sys.modules["oracle.pcg"] = saved
        oracle.pcg = saved
