"""Pins for the CPU oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to something independent of its own code: dense
brute force on tiny inputs, matrix identities, a closed form (the 13-point
stencil of the squared 5-point Laplacian; the C-hat size formula), the worked
example printed in gMAGNUS Fig. 1, the chunk counts printed in Tables V/VI, and
the partition and nesting properties any column-range split must have.
"""
import json
import os

import numpy as np
import pytest

import oracle
from sparse_gemm_irregular_gm_gb300 import inputs as gi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dense(M) -> np.ndarray:
    D = np.zeros((M.n_rows, M.n_cols))
    r = np.repeat(np.arange(M.n_rows), np.diff(M.row_ptr))
    np.add.at(D, (r, M.col), M.val)
    return D


def pattern(M) -> np.ndarray:
    P = np.zeros((M.n_rows, M.n_cols), dtype=np.int64)
    r = np.repeat(np.arange(M.n_rows), np.diff(M.row_ptr))
    P[r, M.col] = 1
    return P


def oracle_dense(C, n_rows, n_cols):
    D = np.zeros((n_rows, n_cols))
    S = np.zeros((n_rows, n_cols), dtype=bool)
    for s, i in enumerate(C.rows):
        lo, hi = C.row_ptr[s], C.row_ptr[s + 1]
        D[i, C.col[lo:hi]] = C.val[lo:hi]
        S[i, C.col[lo:hi]] = True
    return D, S


def assert_rows_sorted_unique(C):
    for s in range(C.rows.size):
        c = C.col[C.row_ptr[s]:C.row_ptr[s + 1]]
        assert np.all(np.diff(c) > 0)


def canonical(M):
    """Sorted, duplicate-summed copy of M (explicit zeros kept)."""
    r = np.repeat(np.arange(M.n_rows), np.diff(M.row_ptr))
    key = r.astype(np.int64) * M.n_cols + M.col
    uk, inv = np.unique(key, return_inverse=True)
    v = np.zeros(uk.size)
    np.add.at(v, inv, M.val)
    rr = uk // M.n_cols
    rp = np.zeros(M.n_rows + 1, dtype=np.int64)
    np.cumsum(np.bincount(rr, minlength=M.n_rows), out=rp[1:])
    return rp, (uk % M.n_cols).astype(np.int32), v


# --- dense brute force -------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("shape", [(7, 5, 9), (16, 16, 16), (33, 20, 41), (1, 64, 3), (64, 1, 64)])
def test_oracle_matches_dense_bruteforce(seed, shape):
    m, k, n = shape
    A = gi.random_csr(m, k, 0.3, seed, values="int", unsorted=True, duplicates=True,
                      explicit_zeros=True, empty_rows=0.2)
    B = gi.random_csr(k, n, 0.25, seed + 100, values="int", unsorted=True, duplicates=True,
                      explicit_zeros=True, empty_rows=0.2)
    C = oracle.spgemm(A, B)
    assert_rows_sorted_unique(C)
    D, S = oracle_dense(C, m, n)
    # Integer-valued fp64 products and sums are exact here.
    np.testing.assert_array_equal(D, dense(A) @ dense(B))
    # Structure: (i, j) stored iff some stored A[i,k] meets a stored B[k,j].
    np.testing.assert_array_equal(S, (pattern(A) @ pattern(B)) > 0)
    # abs scale is sum |a*b| over the same pairs (each stored duplicate counted).
    Dabs, _ = oracle_dense(oracle.OracleC(C.rows, n, C.row_ptr, C.col, C.abs_scale, C.abs_scale), m, n)
    np.testing.assert_array_equal(Dabs, _abs_pairs(A, B))


def _abs_pairs(A, B):
    # sum over stored pairs of |a*b| (duplicates counted separately), by brute force
    out = np.zeros((A.n_rows, B.n_cols))
    for i in range(A.n_rows):
        for p in range(A.row_ptr[i], A.row_ptr[i + 1]):
            j = A.col[p]
            for q in range(B.row_ptr[j], B.row_ptr[j + 1]):
                out[i, B.col[q]] += abs(A.val[p] * B.val[q])
    return out


def test_oracle_empty_operands():
    A = gi.random_csr(5, 4, 0.0, 1)
    B = gi.random_csr(4, 6, 0.5, 2)
    C = oracle.spgemm(A, B)
    assert C.nnz == 0 and C.row_ptr.tolist() == [0] * 6
    C = oracle.spgemm(B.__class__(0, 4, np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0)), B)
    assert C.rows.size == 0 and C.nnz == 0


def test_oracle_dimension_mismatch_and_bad_index():
    A = gi.random_csr(5, 4, 0.5, 1)
    B = gi.random_csr(5, 6, 0.5, 2)
    with pytest.raises(ValueError):
        oracle.spgemm(A, B)
    B2 = gi.random_csr(4, 6, 0.5, 2)
    A.col[0] = 9
    with pytest.raises(ValueError):
        oracle.spgemm(A, B2)
    with pytest.raises(ValueError):
        oracle.ip_counts(A, B2)


# --- identities and permutations --------------------------------------------

def test_oracle_identity():
    A = gi.random_csr(40, 30, 0.2, 7, values="uniform", unsorted=True, duplicates=True, explicit_zeros=True)
    rp, col, val = canonical(A)
    C = oracle.spgemm(A, gi.identity(30))
    np.testing.assert_array_equal(C.row_ptr, rp)
    np.testing.assert_array_equal(C.col, col)
    np.testing.assert_allclose(C.val, val, rtol=1e-15, atol=0)
    C = oracle.spgemm(gi.identity(40), A)
    np.testing.assert_array_equal(C.row_ptr, rp)
    np.testing.assert_array_equal(C.col, col)
    np.testing.assert_allclose(C.val, val, rtol=1e-15, atol=0)


def test_oracle_row_and_column_permutations():
    rng = np.random.default_rng(3)
    A = gi.random_csr(50, 35, 0.15, 11, values="uniform")
    B = gi.random_csr(35, 45, 0.15, 12, values="uniform")
    C = oracle.spgemm(A, B)
    # (P A) B = P (A B): row i of the product is row perm[i] of A B.
    perm = rng.permutation(50)
    PA_rp, PA_col, PA_val = _permute_rows(A, perm)
    PA = gi.CSR(50, 35, PA_rp, PA_col, PA_val)
    C2 = oracle.spgemm(PA, B)
    for i in range(50):
        s = perm[i]
        np.testing.assert_array_equal(C2.col[C2.row_ptr[i]:C2.row_ptr[i + 1]], C.col[C.row_ptr[s]:C.row_ptr[s + 1]])
        np.testing.assert_array_equal(C2.val[C2.row_ptr[i]:C2.row_ptr[i + 1]], C.val[C.row_ptr[s]:C.row_ptr[s + 1]])
    # A (B Q): column k of A B moves to column q[k].
    q = rng.permutation(45)
    BQ = gi.CSR(35, 45, B.row_ptr.copy(), q[B.col].astype(np.int32), B.val.copy())
    C3 = oracle.spgemm(A, BQ)
    for i in range(50):
        c = C.col[C.row_ptr[i]:C.row_ptr[i + 1]]
        v = C.val[C.row_ptr[i]:C.row_ptr[i + 1]]
        order = np.argsort(q[c])
        np.testing.assert_array_equal(C3.col[C3.row_ptr[i]:C3.row_ptr[i + 1]], q[c][order])
        np.testing.assert_array_equal(C3.val[C3.row_ptr[i]:C3.row_ptr[i + 1]], v[order])


def _permute_rows(A, perm):
    lens = np.diff(A.row_ptr)[perm]
    rp = np.zeros(A.n_rows + 1, dtype=np.int64)
    np.cumsum(lens, out=rp[1:])
    col = np.concatenate([A.col[A.row_ptr[s]:A.row_ptr[s + 1]] for s in perm]).astype(np.int32)
    val = np.concatenate([A.val[A.row_ptr[s]:A.row_ptr[s + 1]] for s in perm])
    return rp, col, val


def test_oracle_row_subset_equals_full():
    A = gi.rmat(9, 8, seed=5)
    C = oracle.spgemm(A, A)
    rows = np.array([0, 3, 511, 17, 17, 200], dtype=np.int64)
    S = oracle.spgemm_rows(A, A, rows)
    for s, i in enumerate(rows):
        np.testing.assert_array_equal(S.col[S.row_ptr[s]:S.row_ptr[s + 1]], C.col[C.row_ptr[i]:C.row_ptr[i + 1]])
        np.testing.assert_array_equal(S.val[S.row_ptr[s]:S.row_ptr[s + 1]], C.val[C.row_ptr[i]:C.row_ptr[i + 1]])


# --- closed forms -------------------------------------------------------------

def laplacian_square_closed_form(nx, ny):
    """A^2 for the 5-point Laplacian A = 4I - (grid adjacency), entry by entry.

    diag: 16 + deg(p); grid neighbours: -8 (paths p->p->q and p->q->q);
    distance-2 along an axis: 1 (one path); diagonal neighbours: 2 (two paths).
    """
    entries = {}
    for y in range(ny):
        for x in range(nx):
            p = y * nx + x
            deg = sum(0 <= x + dx < nx and 0 <= y + dy < ny for dx, dy in ((1, 0), (-1, 0), (0, 1), (0, -1)))
            row = {p: 16.0 + deg}
            for dx, dy, v in ((1, 0, -8.0), (-1, 0, -8.0), (0, 1, -8.0), (0, -1, -8.0),
                              (2, 0, 1.0), (-2, 0, 1.0), (0, 2, 1.0), (0, -2, 1.0),
                              (1, 1, 2.0), (1, -1, 2.0), (-1, 1, 2.0), (-1, -1, 2.0)):
                if 0 <= x + dx < nx and 0 <= y + dy < ny:
                    row[(y + dy) * nx + x + dx] = v
            entries[p] = row
    return entries


@pytest.mark.parametrize("nx,ny", [(1, 1), (2, 3), (7, 5), (24, 17)])
def test_oracle_laplacian_square_closed_form(nx, ny):
    A = gi.laplacian_2d(nx, ny)
    C = oracle.spgemm(A, A)
    ref = laplacian_square_closed_form(nx, ny)
    for i in range(nx * ny):
        cols = C.col[C.row_ptr[i]:C.row_ptr[i + 1]].tolist()
        vals = C.val[C.row_ptr[i]:C.row_ptr[i + 1]].tolist()
        assert cols == sorted(ref[i])
        assert vals == [ref[i][c] for c in cols]


def test_laplacian_1024_nnz_closed_form():
    # Count of the clipped 13-point stencil on a 1024 x 1024 grid, per offset class.
    n = 1024
    count = n * n                      # diagonal
    count += 4 * n * (n - 1)           # axis neighbours
    count += 4 * n * (n - 2)           # distance 2 along an axis
    count += 4 * (n - 1) * (n - 1)     # diagonal neighbours
    assert count == 13_611_012


@pytest.mark.parametrize("seed", [1, 2])
def test_ip_counts_closed_form(seed):
    A = gi.rmat(10, 8, seed=seed)
    B = gi.rmat(10, 4, seed=seed + 10)
    u = oracle.ip_counts(A, B)
    # Sum over rows = sum over k of nnz(A[:,k]) * nnz(B[k,:]) (C-hat size; gMAGNUS
    # Sec. III-B slice sizes, SparseDitto SpGEMM Eq. (1)).
    col_counts = np.bincount(A.col, minlength=A.n_cols).astype(np.int64)
    assert int(u.sum()) == int((col_counts * np.diff(B.row_ptr)).sum())
    # Per row, u(i) is the number of products the expansion emits.
    rows = np.arange(0, A.n_rows, 37)
    ex = oracle.expand_rows(A, B, rows)
    assert [len(e) for e in ex] == u[rows].tolist()
    # nnz(C[i,:]) <= u(i), equality iff no two products share a column.
    C = oracle.spgemm(A, B)
    assert np.all(np.diff(C.row_ptr) <= u)


# --- gMAGNUS Fig. 1 worked example -----------------------------------------

def _fig1():
    with open(os.path.join(GOLDEN, "fig1_worked_example.json")) as f:
        g = json.load(f)
    rng = np.random.default_rng(42)
    syms = {}

    def sym(name):
        if name not in syms:
            syms[name] = float(rng.integers(2, 50)) + rng.random()
        return syms[name]

    def build(rows, shape):
        n, m = shape
        rp = [0]
        col, val = [], []
        for i in range(n):
            for c, s in rows.get(str(i), []):
                col.append(c)
                val.append(sym(s))
            rp.append(len(col))
        return gi.CSR(n, m, np.array(rp, np.int64), np.array(col, np.int32), np.array(val, np.float64))

    A = build(g["A_rows"], g["A_shape"])
    B = build(g["B_rows"], g["B_shape"])

    def prod(label):  # "A11B10" -> value of A11 * value of B10
        return sym(label[:3]) * sym(label[3:])

    return g, A, B, prod


def test_fig1_expansion_and_reorder():
    g, A, B, prod = _fig1()
    ex = oracle.expand_rows(A, B, g["heavy_rows"])
    for items, cols, labels in zip(ex, g["Chat_col"], g["Chat_val"]):
        assert sorted(items) == sorted(zip(cols, [prod(s) for s in labels]))
    k = 0
    for items in ex:
        for ch in oracle.split_chunks(items, g["n_chunks"], g["chunk_width"]):
            assert sorted(ch) == sorted(zip(g["Creord_col"][k], [prod(s) for s in g["Creord_val"][k]]))
            k += 1
    assert k == len(g["Creord_col"])


def test_fig1_result():
    g, A, B, prod = _fig1()
    C = oracle.spgemm(A, B)
    for r, entries in g["C_rows"].items():
        i = int(r)
        cols = C.col[C.row_ptr[i]:C.row_ptr[i + 1]].tolist()
        vals = C.val[C.row_ptr[i]:C.row_ptr[i + 1]].tolist()
        assert cols == [c for c, _ in entries]
        for v, (_, labels) in zip(vals, entries):
            assert v == pytest.approx(sum(prod(s) for s in labels), rel=1e-15)
    # Heavy rows under a threshold below both row sizes (u = 7 and 3).
    u = oracle.ip_counts(A, B)
    assert u.tolist() == [0, 7, 3]
    heavy, light = oracle.thresh_partition(u, 2)
    assert heavy.tolist() == g["heavy_rows"] and light.tolist() == [0]
    p = oracle.magnus_params(g["C_m"], dense_width=4, n_chunks_max=2, tau=2)
    assert p.v_chunks == [g["n_chunks"]] and p.widths == [g["chunk_width"]]


def test_heavy_means_exceeding_tau():
    """A row is heavy only when its products exceed tau (gMAGNUS Sec. I and
    Sec. II-B: the rows whose intermediate products do not fit the local-memory
    accumulator of capacity tau). A row with exactly tau products still fits, so
    it is light; a ">=" test would call it heavy. The Fig. 1 rows have u = 7 and
    u = 3, so tau = 3 and tau = 7 each put one row exactly on the threshold."""
    g, A, B, _ = _fig1()
    u = oracle.ip_counts(A, B)
    assert u.tolist() == [0, 7, 3]
    heavy, light = oracle.thresh_partition(u, 3)
    assert heavy.tolist() == [1] and light.tolist() == [0, 2]
    heavy, light = oracle.thresh_partition(u, 7)
    assert heavy.tolist() == [] and light.tolist() == [0, 1, 2]
    heavy, light = oracle.thresh_partition(u, 6)
    assert heavy.tolist() == [1] and light.tolist() == [0, 2]
    # every row lands in exactly one of the two lists, order preserved
    for tau in range(0, 9):
        heavy, light = oracle.thresh_partition(u, tau)
        assert sorted(heavy.tolist() + light.tolist()) == [0, 1, 2]
        assert heavy.tolist() == sorted(heavy.tolist()) and light.tolist() == sorted(light.tolist())


# --- intermediate matrices: C-hat and the chunk split, on random inputs ---------

@pytest.mark.parametrize("seed", range(4))
def test_expand_rows_against_dense_and_counts(seed):
    """C-hat rows (Sec. II-C Eq. (2)): row i holds u(i) elements (the count of
    the C-hat size formula), and summing its elements by column gives row i of
    the dense product A @ B, over exactly the columns the pattern product
    reaches."""
    A = gi.random_csr(12, 15, 0.3, seed, values="int", unsorted=True, duplicates=True, empty_rows=0.2)
    B = gi.random_csr(15, 40, 0.25, seed + 100, values="int", unsorted=True, duplicates=True, empty_rows=0.2)
    rows = list(range(A.n_rows))
    ex = oracle.expand_rows(A, B, rows)
    u = oracle.ip_counts(A, B)
    D = dense(A) @ dense(B)
    reach = (pattern(A) @ pattern(B)) > 0
    for i, items in zip(rows, ex):
        assert len(items) == u[i]
        acc = np.zeros(B.n_cols)
        seen = np.zeros(B.n_cols, dtype=bool)
        for c, v in items:
            acc[c] += v
            seen[c] = True
        np.testing.assert_array_equal(seen, reach[i])
        np.testing.assert_array_equal(acc, D[i])


@pytest.mark.parametrize("seed", range(4))
def test_split_chunks_partitions_a_row(seed):
    """The chunk split (Sec. III-C): every element lands in the chunk of its
    column range with a chunk-local column below the width, nothing is lost or
    duplicated, and restoring c * width + local gives the row back."""
    rng = np.random.default_rng(seed)
    width, n_chunks = 16, 8
    items = [(int(c), float(v)) for c, v in zip(rng.integers(0, width * n_chunks, 300), rng.normal(size=300))]
    chunks = oracle.split_chunks(items, n_chunks, width)
    assert len(chunks) == n_chunks
    assert sum(len(ch) for ch in chunks) == len(items)
    back = []
    for c, ch in enumerate(chunks):
        for local, v in ch:
            assert 0 <= local < width
            back.append((c * width + local, v))
    assert sorted(back) == sorted(items)
    with pytest.raises(ValueError):
        oracle.split_chunks([(width * n_chunks, 1.0)], n_chunks, width)


def test_split_chunks_two_levels_equal_one_finer_split():
    """Hierarchy of chunks (Fig. 1, Sec. III-C): splitting a row into v0 chunks
    of width w0 and each of those into v1 chunks of width w0 / v1 yields the same
    element sets, with the same local columns, as one split into v0 * v1 chunks of
    width w0 / v1, chunk c0 * v1 + c1."""
    rng = np.random.default_rng(7)
    v0, v1, w1 = 4, 8, 32
    w0 = v1 * w1
    items = [(int(c), float(i)) for i, c in enumerate(rng.integers(0, v0 * w0, 2000))]
    fine = oracle.split_chunks(items, v0 * v1, w1)
    for c0, ch in enumerate(oracle.split_chunks(items, v0, w0)):
        for c1, sub in enumerate(oracle.split_chunks(ch, v1, w1)):
            assert sorted(sub) == sorted(fine[c0 * v1 + c1])


# --- the row split over several GPUs -------------------------------------------

def test_row_split_worked_cases():
    """Hand-worked splits. u = [5, 0, 3, 8, 2, 2] (T = 20), two parts: the target
    10 lies between S(3) = 8 and S(4) = 16, nearer 8, so rows [0, 3) and [3, 6)
    (8 and 12 products). Equal rows split evenly; no products split rows evenly;
    one giant row stays alone."""
    assert oracle.row_split([5, 0, 3, 8, 2, 2], 2).tolist() == [0, 3, 6]
    assert oracle.row_split([1] * 10, 5).tolist() == [0, 2, 4, 6, 8, 10]
    assert oracle.row_split([0, 0, 0], 2).tolist() == [0, 1, 3]
    assert oracle.row_split([100, 1, 1, 1], 3).tolist() == [0, 0, 1, 4]
    assert oracle.row_split([7], 1).tolist() == [0, 1]
    assert oracle.row_split([], 3).tolist() == [0, 0, 0, 0]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("n_parts", [1, 2, 3, 8])
def test_row_split_balances_products(seed, n_parts):
    """Every split covers the rows once, in order, and no part is further from
    T / n_parts than the largest row's products (each bound sits next to its
    target); on R-MAT row counts, against a brute-force search over all bounds of
    the best achievable balance for two parts."""
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 50, 40) * (rng.random(40) < 0.8)
    b = oracle.row_split(u, n_parts)
    assert b[0] == 0 and b[-1] == u.size and np.all(np.diff(b) >= 0)
    T = int(u.sum())
    parts = [int(u[b[q]:b[q + 1]].sum()) for q in range(n_parts)]
    assert sum(parts) == T
    S = np.concatenate([[0], np.cumsum(u)])
    for q in range(1, n_parts):  # each bound is at most one row away from its target
        assert abs(n_parts * S[b[q]] - q * T) <= n_parts * max(int(u.max()), 0)
    if n_parts == 2:
        best = min(abs(2 * int(S[r]) - T) for r in range(u.size + 1))
        assert abs(2 * int(S[b[1]]) - T) == best
