"""CPU oracle for the gMAGNUS SpGEMM C = A*B (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. It shares no code with the CUDA library and never
imports it; both sides are fed by the seeded generators in
``sparse_gemm_irregular_gm_gb300.inputs``.

Contents and what each follows (gMAGNUS, "Fast SpGEMM on GPUs for Irregular
Matrices via Hierarchical Multisplit"):

* ``spgemm`` / ``spgemm_rows`` -- Gustavson, Sec. II-B Eq. (1) and Algorithm 1,
  in ``gm_oracle.cpp`` (std::map accumulator per row, OpenMP over rows).
* ``ip_counts``        -- per-row intermediate-product count u(i), Sec. III-A
  (InterOffsets); the same closed form is SparseDitto "SpGEMM" Eq. (1).
* ``thresh_partition`` -- heavy rows are those whose u(i) exceeds tau, Sec. III-A
  (Algorithm 3, ThreshPartition), order preserved.
* ``row_split``        -- consecutive row ranges of about equal intermediate
  products, for one product spread over several GPUs (not in the pages, which
  run on one GPU; the balance follows the u(i) of Sec. III-A).
* ``magnus_params``    -- Sec. III-D, Eqs. (4)-(7): tau, dense width, required
  and maximum chunk counts, number of levels and chunks per level.
* ``expand_rows``      -- the intermediate matrix C-hat of the heavy rows as a
  multiset per row: every product A[i,j]*B[j,k] with column k (Sec. II-C,
  Eq. (2); Fig. 1 "Outer product").
* ``split_chunks``     -- one multisplit level: the elements of a row whose
  column falls in [c*w, (c+1)*w) form chunk c, with the column shifted to
  col - c*w (Sec. III-A, Fig. 1 "Reorder"; Sec. III-C, GetChunk).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gm_oracle.cpp")
_LIB = os.path.join(_HERE, "libgm_oracle.so")
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile gm_oracle.cpp into libgm_oracle.so next to it (host gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC",
                               _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.gm_oracle_ip_counts.restype = ctypes.c_int
        lib.gm_oracle_ip_counts.argtypes = [ctypes.c_int64, _i64p, _i32p, ctypes.c_int64, _i64p, _i64p]
        lib.gm_oracle_spgemm_rows.restype = ctypes.c_void_p
        lib.gm_oracle_spgemm_rows.argtypes = [
            ctypes.c_int64, ctypes.c_int64, _i64p, _i32p, _f64p,
            ctypes.c_int64, ctypes.c_int64, _i64p, _i32p, _f64p,
            _i64p, ctypes.c_int64, ctypes.c_int]
        lib.gm_oracle_result_rows.restype = ctypes.c_int64
        lib.gm_oracle_result_rows.argtypes = [ctypes.c_void_p]
        lib.gm_oracle_result_nnz.restype = ctypes.c_int64
        lib.gm_oracle_result_nnz.argtypes = [ctypes.c_void_p]
        lib.gm_oracle_result_copy.restype = None
        lib.gm_oracle_result_copy.argtypes = [ctypes.c_void_p, _i64p, _i32p, _f64p, _f64p]
        lib.gm_oracle_result_free.restype = None
        lib.gm_oracle_result_free.argtypes = [ctypes.c_void_p]
        lib.gm_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def max_threads() -> int:
    return int(_load().gm_oracle_max_threads())


def ip_counts(A, B) -> np.ndarray:
    """u(i) = sum over stored A[i,j] of nnz(B[j,:]) for every row i of A."""
    lib = _load()
    u = np.zeros(A.n_rows, dtype=np.int64)
    rc = lib.gm_oracle_ip_counts(A.n_rows, _p(A.row_ptr, _i64p), _p(A.col, _i32p),
                                 B.n_rows, _p(B.row_ptr, _i64p), _p(u, _i64p))
    if rc != 0:
        raise ValueError("column index of A out of range")
    return u


@dataclass
class OracleC:
    """Rows of C in CSR form; ``rows`` are the row ids of A they belong to."""

    rows: np.ndarray
    n_cols: int
    row_ptr: np.ndarray
    col: np.ndarray
    val: np.ndarray
    abs_scale: np.ndarray  # sum_j |A[i,j]*B[j,k]| per stored entry

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])


def spgemm_rows(A, B, rows=None, threads: int = 0) -> OracleC:
    """C[rows,:] = A[rows,:] @ B by Gustavson (all rows when ``rows`` is None)."""
    lib = _load()
    if A.n_cols != B.n_rows:
        raise ValueError("inner dimensions differ")
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    h = lib.gm_oracle_spgemm_rows(
        A.n_rows, A.n_cols, _p(A.row_ptr, _i64p), _p(A.col, _i32p), _p(A.val, _f64p),
        B.n_rows, B.n_cols, _p(B.row_ptr, _i64p), _p(B.col, _i32p), _p(B.val, _f64p),
        None if sel is None else _p(sel, _i64p), 0 if sel is None else sel.size, int(threads))
    if not h:
        raise ValueError("index out of range in A or B")
    try:
        n = lib.gm_oracle_result_rows(h)
        nnz = lib.gm_oracle_result_nnz(h)
        rp = np.empty(n + 1, dtype=np.int64)
        col = np.empty(nnz, dtype=np.int32)
        val = np.empty(nnz, dtype=np.float64)
        absv = np.empty(nnz, dtype=np.float64)
        lib.gm_oracle_result_copy(h, _p(rp, _i64p), _p(col, _i32p), _p(val, _f64p), _p(absv, _f64p))
    finally:
        lib.gm_oracle_result_free(h)
    row_ids = np.arange(A.n_rows, dtype=np.int64) if sel is None else sel
    return OracleC(row_ids, B.n_cols, rp, col, val, absv)


def spgemm(A, B, threads: int = 0) -> OracleC:
    return spgemm_rows(A, B, None, threads)


# ---------------------------------------------------------------------------
# Heavy/light partition (Sec. III-A, Algorithm 3 lines 3-4)
# ---------------------------------------------------------------------------

def thresh_partition(u: np.ndarray, tau: int):
    """Row ids with u > tau (heavy) and the rest (light), each in increasing order.

    A row is heavy when its intermediate products exceed the capacity tau of the
    local-memory accumulator (Sec. I; Sec. II-B "heavy rows").
    """
    u = np.asarray(u)
    heavy = np.nonzero(u > tau)[0].astype(np.int64)
    light = np.nonzero(u <= tau)[0].astype(np.int64)
    return heavy, light


# ---------------------------------------------------------------------------
# Row split over several GPUs (the pages run on one GPU; see row_split)
# ---------------------------------------------------------------------------

def row_split(u: np.ndarray, n_parts: int) -> np.ndarray:
    """Bounds of n_parts consecutive row ranges with about equal products.

    The pages measure one GPU only; spreading one product over several takes a
    split of A's rows, and the plainest one balances the quantity the method's
    work follows, the intermediate products u(i) of each row (Sec. III-A). With
    S(r) = u(0) + ... + u(r-1) and T = S(n): bounds[0] = 0, bounds[n_parts] = n,
    and bounds[q] is the r at which n_parts * S(r) is nearest to q * T, taken
    between the last r below q * T and the first r reaching it (the lower one on
    a tie). Without products the rows are split evenly: q * n // n_parts.
    Exact integer arithmetic (Python ints)."""
    u = [int(x) for x in np.asarray(u, dtype=np.int64)]
    n = len(u)
    S = [0]
    for x in u:
        S.append(S[-1] + x)
    T = S[-1]
    bounds = [0]
    for q in range(1, n_parts):
        if T == 0:
            bounds.append(q * n // n_parts)
            continue
        want = q * T
        first = next(r for r in range(n + 1) if n_parts * S[r] >= want)
        below, above = want - n_parts * S[first - 1], n_parts * S[first] - want
        bounds.append(first - 1 if below <= above else first)
    bounds.append(n)
    return np.asarray(bounds, dtype=np.int64)


# ---------------------------------------------------------------------------
# Parameter selection (Sec. III-D, Eqs. (4)-(7))
# ---------------------------------------------------------------------------

def _floor_pow2(x: int) -> int:
    if x < 1:
        raise ValueError("no power of two below 1")
    return 1 << (int(x).bit_length() - 1)


def _next_pow2(x: int) -> int:
    x = max(1, int(x))
    return 1 << (x - 1).bit_length()


def _log2_exact(x: int) -> int:
    assert x >= 1 and (x & (x - 1)) == 0
    return x.bit_length() - 1


@dataclass
class MagnusParams:
    s_lm: int
    tau: int
    n_dense_numeric: int          # s_LM / (s_val + s_bitMap), before rounding
    dense_width: int              # n_denseNumeric floored to a power of two
    n_chunks_required: int
    n_min_group_elems: int
    n_group_rows: int
    n_chunks_max_raw: int         # Eq. (5) solved for n_chunksMax, before rounding
    n_chunks_max: int
    n_levels: int
    v_chunks: list = field(default_factory=list)
    widths: list = field(default_factory=list)  # column width of a chunk after each level


def magnus_params(c_m: int, s_lm: int = 232448, s_col: int = 4, s_val: int = 8,
                  s_rowptr: int = 8, s_histo: int = 4, s_bitmap: int = 1,
                  n_subgroups: int = 32, alpha: int = 2,
                  dense_width: int | None = None, n_chunks_max: int | None = None,
                  tau: int | None = None) -> MagnusParams:
    """GetMagnusParams(C.m, s_LM) of Sec. III-D, all divisions floored.

    Readings of the extracted text (the formulas are partly garbled there):
      * Eq. (4): tau = s_LM / (alpha * (s_C.col + s_C.val)): the hash map holds
        alpha*tau (key, value) slots in s_LM bytes.
      * n_denseNumeric = s_LM / (s_C.val + s_bitMap) is floored to a power of two.
      * n_chunksRequired = ceil(C.m / n_denseNumeric) is rounded UP to a power of
        two, so that the last-level chunk is never wider than the dense array.
      * Eq. (5) is solved for n_chunksMax (Eq. (6) is its solution) and the
        result floored to a power of two; n_minGroupElems = s_LM / (2(s_col+s_val))
        and n_groupRows = ceil((n_minGroupElems - 1) / tau) + 1.
      * Eq. (7): n_levels = ceil(log2 n_chunksRequired / log2 n_chunksMax); one
        level when n_chunksRequired <= n_chunksMax; none when it is 1.
      * v_chunks[i] = n_chunksMax for every level but the last, and the last is
        n_chunksRequired / n_chunksMax^(n_levels-1) (a quotient).
    ``dense_width``, ``n_chunks_max`` and ``tau`` override the derived values
    (the chunk tables of Sec. IV-B come from other hardware budgets).
    """
    t = s_lm // (alpha * (s_col + s_val)) if tau is None else int(tau)
    n_dense = s_lm // (s_val + s_bitmap)
    d = _floor_pow2(n_dense) if dense_width is None else int(dense_width)
    req = _next_pow2(-(-int(c_m) // d))
    n_min_ge = s_lm // (2 * (s_col + s_val))
    n_gr = -(-(n_min_ge - 1) // t) + 1
    ncm_raw = (s_lm - n_min_ge * (s_col + s_val) - s_histo) // (n_gr * n_subgroups * s_histo + s_rowptr * n_gr)
    ncm = _floor_pow2(ncm_raw) if n_chunks_max is None else int(n_chunks_max)
    if req == 1:
        levels, v = 0, []
    elif req <= ncm:
        levels, v = 1, [req]
    else:
        lr, lm = _log2_exact(req), _log2_exact(ncm)
        levels = -(-lr // lm)
        v = [ncm] * (levels - 1) + [req // ncm ** (levels - 1)]
    widths, w = [], d * req
    for c in v:
        w //= c
        widths.append(w)
    return MagnusParams(s_lm, t, n_dense, d, req, n_min_ge, n_gr, ncm_raw, ncm, levels, v, widths)


# ---------------------------------------------------------------------------
# Intermediate matrices (Sec. II-C Eq. (2), Sec. III-A Fig. 1, Sec. III-C)
# ---------------------------------------------------------------------------

def expand_rows(A, B, rows):
    """C-hat restricted to ``rows``: for each row, the list of (column, product).

    Every stored A[i,j] contributes A[i,j]*B[j,k] at column k for every stored
    B[j,k]; the list is a multiset (order is not part of the definition).
    Pure-Python loops: small cases only.
    """
    out = []
    for i in rows:
        items = []
        for p in range(int(A.row_ptr[i]), int(A.row_ptr[i + 1])):
            j = int(A.col[p])
            for q in range(int(B.row_ptr[j]), int(B.row_ptr[j + 1])):
                items.append((int(B.col[q]), float(A.val[p]) * float(B.val[q])))
        out.append(items)
    return out


def split_chunks(row_items, n_chunks: int, width: int):
    """Split one row's (column, value) multiset into ``n_chunks`` column ranges.

    Chunk c holds the elements with c*width <= column < (c+1)*width, stored with
    the chunk-local column (column - c*width).
    """
    chunks = [[] for _ in range(n_chunks)]
    for col, v in row_items:
        c = col // width
        if not 0 <= c < n_chunks:
            raise ValueError("column outside the split range")
        chunks[c].append((col - c * width, v))
    return chunks
