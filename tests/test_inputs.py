"""The seeded generators produce the shapes and structure they promise."""
import numpy as np

from sparse_gemm_irregular_gm_gb300 import inputs as gi


def test_rmat_deterministic_and_valid():
    A = gi.rmat(10, 8, seed=1)
    B = gi.rmat(10, 8, seed=1)
    assert A.n_rows == A.n_cols == 1024
    assert np.array_equal(A.col, B.col) and np.array_equal(A.val, B.val)
    assert 0 < A.nnz <= 8 * 1024
    for i in range(A.n_rows):  # rows sorted, duplicates collapsed
        assert np.all(np.diff(A.col[A.row_ptr[i]:A.row_ptr[i + 1]]) > 0)
    assert A.val.min() >= -1.0 and A.val.max() < 1.0
    # power law: quadrant a (top-left) is the densest, so low rows hold most entries
    lens = np.diff(A.row_ptr)
    assert lens[:512].sum() > 2 * lens[512:].sum()
    Ai = gi.rmat(10, 8, seed=1, values="int")
    assert np.array_equal(Ai.col, A.col)
    assert set(np.unique(Ai.val)) <= set(range(-3, 4)) and 0.0 in set(Ai.val)


def test_laplacian_structure():
    A = gi.laplacian_2d(1024)
    assert A.n_rows == 1 << 20 and A.nnz == 5 * (1 << 20) - 4 * 1024
    small = gi.laplacian_2d(4, 3)
    D = np.zeros((12, 12))
    r = np.repeat(np.arange(12), np.diff(small.row_ptr))
    D[r, small.col] = small.val
    assert np.all(np.diag(D) == 4) and np.allclose(D, D.T)
    assert D[0, 1] == -1 and D[0, 4] == -1 and D[3, 4] == 0  # no wrap-around


def test_erdos_renyi_distinct_columns():
    A = gi.erdos_renyi(1 << 12, 8, seed=1)
    cols = A.col.reshape(-1, 8)
    assert np.all(np.diff(cols, axis=1) > 0)
    assert A.nnz == 8 << 12


def test_random_csr_options():
    A = gi.random_csr(30, 20, 0.3, 1, unsorted=True, duplicates=True, explicit_zeros=True, empty_rows=0.3)
    A.check()
    assert (np.diff(A.row_ptr) == 0).any()
    assert (A.val == 0).any()


def test_rmat_grid_pair_is_seeded_and_distinct():
    A, B = gi.named_pair("rmatAB_s10_a4_b8", seed=3)
    A2, B2 = gi.rmat_pair(10, 4, 8, seed=3)
    assert A.n_rows == B.n_rows == A.n_cols == B.n_cols == 1024
    np.testing.assert_array_equal(A.col, A2.col)
    np.testing.assert_array_equal(B.val, B2.val)
    assert 3.0 < A.nnz / A.n_rows <= 4.0 and 6.0 < B.nnz / B.n_rows <= 8.0
    assert A.nnz != B.nnz or not np.array_equal(A.col, B.col)
