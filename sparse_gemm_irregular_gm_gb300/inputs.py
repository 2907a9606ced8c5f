"""Seeded synthetic CSR inputs shared by the tests, the benchmark and the oracle.

This module only draws matrices. It holds none of the SpGEMM arithmetic, imports
nothing else from this package, and depends on numpy alone, so that both the
CUDA path and the CPU oracle can be fed the very same arrays.

Workloads (gMAGNUS, "Fast SpGEMM on GPUs for Irregular Matrices via
Hierarchical Multisplit", Sec. IV-A: recursive power-law matrices with the
Graph500 parameters a = 0.57, b = c = 0.19), plus a banded and a uniform one:

* ``rmat``        -- recursive power-law (R-MAT) graph, duplicates collapsed.
* ``laplacian_2d``-- 5-point Laplacian on an nx-by-ny grid (4 / -1 stencil).
* ``erdos_renyi`` -- k distinct uniformly random columns per row.
* ``random_csr``  -- tiny irregular matrices for brute-force checks: optional
                     unsorted rows, duplicate entries and explicit zeros.

Layout of every matrix: row_ptr int64[n_rows+1], col int32[nnz], val float64[nnz].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = ["CSR", "rmat", "rmat_pair", "laplacian_2d", "erdos_renyi", "random_csr", "row_slice",
           "identity", "permutation", "named_workload", "named_pair", "WORKLOADS", "PAIRS"]


@dataclass
class CSR:
    """Host CSR matrix: ``row_ptr`` int64, ``col`` int32, ``val`` float64."""

    n_rows: int
    n_cols: int
    row_ptr: np.ndarray
    col: np.ndarray
    val: np.ndarray

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    def check(self) -> "CSR":
        assert self.row_ptr.dtype == np.int64 and self.row_ptr.shape == (self.n_rows + 1,)
        assert self.col.dtype == np.int32 and self.val.dtype == np.float64
        assert self.row_ptr[0] == 0 and self.col.shape == (self.nnz,) == self.val.shape
        assert np.all(np.diff(self.row_ptr) >= 0)
        if self.nnz:
            assert int(self.col.min()) >= 0 and int(self.col.max()) < self.n_cols
        return self


def _from_keys(n_rows: int, n_cols: int, rows: np.ndarray, cols: np.ndarray) -> tuple:
    """Collapse (row, col) pairs to the sorted set of distinct entries."""
    keys = np.sort(rows.astype(np.int64) * np.int64(n_cols) + cols.astype(np.int64))
    if keys.size:
        first = np.empty(keys.size, dtype=bool)
        first[0] = True
        np.not_equal(keys[1:], keys[:-1], out=first[1:])
        keys = keys[first]
    r = keys // n_cols
    c = (keys - r * n_cols).astype(np.int32)
    row_ptr = np.zeros(n_rows + 1, dtype=np.int64)
    np.cumsum(np.bincount(r, minlength=n_rows), out=row_ptr[1:])
    return row_ptr, c


def _values(rng: np.random.Generator, nnz: int, values: str) -> np.ndarray:
    if values == "uniform":
        return rng.uniform(-1.0, 1.0, size=nnz)  # [-1, 1)
    if values == "int":
        return rng.integers(-3, 4, size=nnz).astype(np.float64)  # {-3..3}, 0 included
    if values == "ones":
        return np.ones(nnz, dtype=np.float64)
    raise ValueError(f"unknown value distribution {values!r}")


def rmat(scale: int, edge_factor: int, a: float = 0.57, b: float = 0.19, c: float = 0.19,
         seed: int = 1, values: str = "uniform") -> CSR:
    """R-MAT graph with 2**scale vertices and edge_factor * 2**scale drawn edges.

    Each edge takes ``scale`` independent quadrant choices with probabilities
    (a, b, c, d = 1-a-b-c), top bit first. Quadrant c or d sets the row bit,
    quadrant b or d sets the column bit. No noise, no vertex permutation;
    self-loops are kept. Duplicate edges are collapsed into one stored entry,
    and one value is then drawn per stored entry.
    """
    n = 1 << scale
    m = edge_factor * n
    rng = np.random.default_rng(seed)
    rows = np.zeros(m, dtype=np.int64)
    cols = np.zeros(m, dtype=np.int64)
    ab, abc = a + b, a + b + c
    step = 1 << 22  # bound the temporary arrays
    for lo in range(0, m, step):
        hi = min(m, lo + step)
        r_acc = np.zeros(hi - lo, dtype=np.int64)
        c_acc = np.zeros(hi - lo, dtype=np.int64)
        for _ in range(scale):
            u = rng.random(hi - lo)
            r_bit = u >= ab
            c_bit = ((u >= a) & (u < ab)) | (u >= abc)
            r_acc = (r_acc << 1) | r_bit
            c_acc = (c_acc << 1) | c_bit
        rows[lo:hi] = r_acc
        cols[lo:hi] = c_acc
    row_ptr, col = _from_keys(n, n, rows, cols)
    val = _values(rng, int(row_ptr[-1]), values)
    return CSR(n, n, row_ptr, col, val).check()


def laplacian_2d(nx: int, ny: int | None = None) -> CSR:
    """5-point Laplacian on an nx-by-ny grid: 4 on the diagonal, -1 per grid neighbour.

    Grid point (x, y) is row/column y*nx + x. Rows are sorted by column.
    """
    ny = nx if ny is None else ny
    n = nx * ny
    idx = np.arange(n, dtype=np.int64)
    x = idx % nx
    y = idx // nx
    parts_r, parts_c, parts_v = [], [], []
    for dx, dy, v in ((0, -1, -1.0), (-1, 0, -1.0), (0, 0, 4.0), (1, 0, -1.0), (0, 1, -1.0)):
        ok = (x + dx >= 0) & (x + dx < nx) & (y + dy >= 0) & (y + dy < ny)
        parts_r.append(idx[ok])
        parts_c.append((idx + dx + dy * nx)[ok])
        parts_v.append(np.full(int(ok.sum()), v))
    r = np.concatenate(parts_r)
    c = np.concatenate(parts_c)
    v = np.concatenate(parts_v)
    order = np.lexsort((c, r))
    r, c, v = r[order], c[order], v[order]
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(r, minlength=n), out=row_ptr[1:])
    return CSR(n, n, row_ptr, c.astype(np.int32), v.astype(np.float64)).check()


def erdos_renyi(n: int, k: int = 8, seed: int = 1, values: str = "uniform") -> CSR:
    """n-by-n matrix with exactly k distinct uniformly random columns per row (sorted).

    Columns are drawn without replacement: rows that draw a repeated column
    redraw all k columns until they are distinct.
    """
    assert k <= n
    rng = np.random.default_rng(seed)
    cols = rng.integers(0, n, size=(n, k), dtype=np.int64)
    cols.sort(axis=1)
    bad = np.nonzero((cols[:, 1:] == cols[:, :-1]).any(axis=1))[0] if k > 1 else np.array([], np.int64)
    while bad.size:
        redraw = rng.integers(0, n, size=(bad.size, k), dtype=np.int64)
        redraw.sort(axis=1)
        cols[bad] = redraw
        still = (redraw[:, 1:] == redraw[:, :-1]).any(axis=1)
        bad = bad[still]
    row_ptr = np.arange(0, n * k + 1, k, dtype=np.int64)
    val = _values(rng, n * k, values)
    return CSR(n, n, row_ptr, cols.reshape(-1).astype(np.int32), val).check()


def random_csr(n_rows: int, n_cols: int, density: float, seed: int, values: str = "int",
               unsorted: bool = False, duplicates: bool = False, explicit_zeros: bool = False,
               empty_rows: float = 0.0) -> CSR:
    """Small irregular CSR matrix for brute-force checks.

    ``unsorted`` shuffles each row, ``duplicates`` repeats some entries (the
    product is linear, so repeated entries simply add), ``explicit_zeros``
    sets some stored values to 0, ``empty_rows`` empties that fraction of rows.
    """
    rng = np.random.default_rng(seed)
    mask = rng.random((n_rows, n_cols)) < density
    if empty_rows > 0:
        mask[rng.random(n_rows) < empty_rows] = False
    r, c = np.nonzero(mask)
    if duplicates and r.size:
        pick = rng.random(r.size) < 0.3
        r = np.concatenate([r, r[pick]])
        c = np.concatenate([c, c[pick]])
        order = np.argsort(r, kind="stable")
        r, c = r[order], c[order]
    v = _values(rng, r.size, values)
    if explicit_zeros and r.size:
        v[rng.random(r.size) < 0.2] = 0.0
    row_ptr = np.zeros(n_rows + 1, dtype=np.int64)
    np.cumsum(np.bincount(r, minlength=n_rows), out=row_ptr[1:])
    if unsorted:
        for i in range(n_rows):
            lo, hi = row_ptr[i], row_ptr[i + 1]
            p = rng.permutation(hi - lo) + lo
            c[lo:hi], v[lo:hi] = c[p].copy(), v[p].copy()
    return CSR(n_rows, n_cols, row_ptr, c.astype(np.int32), v.astype(np.float64)).check()


def identity(n: int) -> CSR:
    return CSR(n, n, np.arange(n + 1, dtype=np.int64), np.arange(n, dtype=np.int32),
               np.ones(n, dtype=np.float64))


def permutation(perm: np.ndarray) -> CSR:
    """P with P[i, perm[i]] = 1, so (P @ X)[i, :] = X[perm[i], :]."""
    n = perm.size
    return CSR(n, n, np.arange(n + 1, dtype=np.int64), perm.astype(np.int32),
               np.ones(n, dtype=np.float64))


# The five A*A workloads: (description, generator of A). C = A @ A.
WORKLOADS = {
    "rmat10": ("A*A, R-MAT scale 10, edge factor 8, fp64 U[-1,1)",
               lambda seed=1: rmat(10, 8, seed=seed)),
    "rmat10_int": ("A*A, R-MAT scale 10, edge factor 8, integer values in {-3..3}",
                   lambda seed=1: rmat(10, 8, seed=seed, values="int")),
    "laplace1024": ("A*A, 2D 5-point Laplacian on a 1024x1024 grid",
                    lambda seed=1: laplacian_2d(1024)),
    "er21": ("A*A, Erdos-Renyi 2^21 x 2^21, 8 distinct columns per row, fp64 U[-1,1)",
             lambda seed=1: erdos_renyi(1 << 21, 8, seed=seed)),
    "rmat18": ("A*A, R-MAT scale 18, edge factor 16, fp64 U[-1,1)",
               lambda seed=1: rmat(18, 16, seed=seed)),
    "rmat16": ("A*A, R-MAT scale 16, edge factor 16, fp64 U[-1,1) (small profiling case)",
               lambda seed=1: rmat(16, 16, seed=seed)),
    "rmat20": ("A*A, R-MAT scale 20, edge factor 16, fp64 U[-1,1)",
               lambda seed=1: rmat(20, 16, seed=seed)),
}


def row_slice(M: CSR, lo: int, hi: int) -> CSR:
    """Rows [lo, hi) of M (all columns kept)."""
    a, b = int(M.row_ptr[lo]), int(M.row_ptr[hi])
    return CSR(hi - lo, M.n_cols, (M.row_ptr[lo:hi + 1] - a).astype(np.int64), M.col[a:b].copy(), M.val[a:b].copy())


# Products of two different matrices: (description, generator of (A, B)). C = A @ B.
PAIRS = {
    "rmat20_rows2k": ("A[2^19 : 2^19 + 2048, :] * A, A = R-MAT scale 20, edge factor 16 (profiling case: "
                      "C.m = 2^20 at a few GB)",
                      lambda seed=1: (lambda A: (row_slice(A, 1 << 19, (1 << 19) + 2048), A))(rmat(20, 16, seed=seed))),
    "rmat20_tail64k": ("A[2^20 - 65536 :, :] * A, A = R-MAT scale 20, edge factor 16 (profiling case: the sparse "
                       "end of the matrix, mostly light rows)",
                       lambda seed=1: (lambda A: (row_slice(A, (1 << 20) - 65536, 1 << 20), A))(rmat(20, 16, seed=seed))),
}


def named_workload(name: str, seed: int = 1) -> CSR:
    return WORKLOADS[name][1](seed)


def rmat_pair(scale: int, a_density: int, b_density: int, seed: int = 1, values: str = "uniform"):
    """A and B of the pages' R-MAT grid (gMAGNUS Sec. IV-A: A.nnz/A.n from 4 to 64,
    B.nnz/B.n from 4 to 16, scales 15 to 20): two independent R-MAT matrices of the
    same scale, drawn with edge factors a_density and b_density (A from seed, B
    from seed + 1000003). Duplicate edges collapse, so nnz/n ends a little below
    the edge factor."""
    return (rmat(scale, a_density, seed=seed, values=values),
            rmat(scale, b_density, seed=seed + 1000003, values=values))


def _grid_name(name: str):
    """(scale, a_density, b_density) of a name rmatAB_s<scale>_a<A>_b<B>, else None."""
    parts = name.split("_")
    if len(parts) != 4 or parts[0] != "rmatAB":
        return None
    try:
        return int(parts[1][1:]), int(parts[2][1:]), int(parts[3][1:])
    except ValueError:
        return None


def named_pair(name: str, seed: int = 1):
    """(A, B) of a named product: the A*A workloads give (A, A); rmatAB_s<scale>_a<A>_b<B>
    is the R-MAT grid pair of rmat_pair."""
    if name in PAIRS:
        return PAIRS[name][1](seed)
    grid = _grid_name(name)
    if grid is not None:
        return rmat_pair(*grid, seed=seed)
    A = named_workload(name, seed)
    return A, A
