"""The row split on the GPU (gm_spgemm_row_split, gm_spgemm_analyze_rows,
gm_row_ptr_shift) against the oracle: the library's bounds equal the oracle's
row_split of the oracle's u(i), and the parts of a product computed one after
another on this GPU, shifted and put together, equal the oracle's whole C
(structure bit-exact, fp64 values within 1e-12 * sum|ab|)."""
import numpy as np
import pytest

import oracle
from sparse_gemm_irregular_gm_gb300 import binding, inputs as gi, shard

from tests.gpu_common import assert_matches

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    binding.load()


CASES = [("rmat12", lambda: gi.rmat(12, 8, seed=3)), ("rmat14_int", lambda: gi.rmat(14, 16, seed=4, values="int")),
         ("laplace", lambda: gi.laplacian_2d(120, 90))]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("n_parts", [1, 2, 3, 8])
def test_library_split_equals_the_oracle_split(name, make, n_parts):
    A = make()
    Ad = binding.to_device(A)
    got = binding.gm_spgemm_row_split(Ad, Ad, n_parts)
    np.testing.assert_array_equal(got, oracle.row_split(oracle.ip_counts(A, A), n_parts))


def test_split_of_a_product_without_products():
    A = gi.CSR(7, 5, np.zeros(8, np.int64), np.zeros(0, np.int32), np.zeros(0))
    B = gi.CSR(5, 4, np.zeros(6, np.int64), np.zeros(0, np.int32), np.zeros(0))
    got = binding.gm_spgemm_row_split(binding.to_device(A), binding.to_device(B), 3)
    np.testing.assert_array_equal(got, oracle.row_split(np.zeros(7, np.int64), 3))


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("n_parts", [2, 5])
def test_parts_put_together_equal_the_whole_product(name, make, n_parts):
    """Each part as one rank would run it (its rows through the library, its row
    pointers shifted by the entries of the parts before it), here one after
    another on this GPU; heavy rows included (tau lowered for the small inputs)."""
    A = make()
    Ad = binding.to_device(A)
    cfg = binding.make_config(tau=256) if name != "laplace" else None
    bounds = binding.gm_spgemm_row_split(Ad, Ad, n_parts, cfg)
    ref = oracle.spgemm(A, A)
    base = 0
    for q in range(n_parts):
        r0, r1 = int(bounds[q]), int(bounds[q + 1])
        C, info = binding.spgemm(Ad, Ad, cfg, rows=(r0, r1), return_info=True)
        assert C.n_rows == r1 - r0 and int(C.row_ptr[0]) == 0
        binding.gm_row_ptr_shift(C.row_ptr, base)
        torch.cuda.synchronize()
        rp = C.row_ptr.cpu().numpy()
        np.testing.assert_array_equal(rp, ref.row_ptr[r0:r1 + 1])
        lo, hi = int(ref.row_ptr[r0]), int(ref.row_ptr[r1])
        part = oracle.OracleC(np.arange(r0, r1), A.n_cols, ref.row_ptr[r0:r1 + 1] - lo, ref.col[lo:hi], ref.val[lo:hi],
                              ref.abs_scale[lo:hi])
        assert_matches(part, rp - base, C.col.cpu().numpy(), C.val.cpu().numpy(), exact="int" in name)
        base += C.nnz
    assert base == ref.nnz


def test_shard_module_on_one_rank_is_the_whole_product():
    A = gi.rmat(11, 8, seed=9)
    Ad = binding.to_device(A)
    part = shard.spgemm_row_shard(Ad, Ad)
    assert (part.row_begin, part.row_end, part.base, part.nnz_all) == (0, A.n_rows, 0, [part.C.nnz])
    ref = oracle.spgemm(A, A)
    torch.cuda.synchronize()
    assert_matches(ref, part.C.row_ptr.cpu().numpy(), part.C.col.cpu().numpy(), part.C.val.cpu().numpy())


@pytest.mark.parametrize("rp_dt,col_dt", [(np.int32, np.int32), (np.int64, np.int64), (np.int32, np.int64)])
def test_row_range_with_other_index_types(rp_dt, col_dt):
    A = gi.rmat(11, 8, seed=5, values="int")
    Ad = binding.to_device(A, row_ptr_dtype=rp_dt, col_dtype=col_dt)
    r0, r1 = 300, 1500
    C = binding.spgemm(Ad, Ad, binding.make_config(tau=128), rows=(r0, r1))
    binding.gm_row_ptr_shift(C.row_ptr, 1000)
    torch.cuda.synchronize()
    ref = oracle.spgemm_rows(A, A, np.arange(r0, r1))
    rp = C.row_ptr.cpu().numpy().astype(np.int64)
    assert C.row_ptr.dtype == torch.from_numpy(np.zeros(1, rp_dt)).dtype
    assert_matches(ref, rp - 1000, C.col.cpu().numpy().astype(np.int32), C.val.cpu().numpy(), exact=True)


def test_row_range_and_shift_argument_errors():
    A = gi.rmat(8, 8, seed=1)
    Ad = binding.to_device(A)
    for rows in ((-1, 5), (5, 4), (0, A.n_rows + 1)):
        with pytest.raises(binding.GmError) as e:
            binding.gm_spgemm_analyze(Ad, Ad, rows=rows)
        assert e.value.status == 1
    with pytest.raises(binding.GmError):
        binding.gm_spgemm_row_split(Ad, Ad, 0)
    rp32 = torch.tensor([0, 5, 2 ** 31 - 10], dtype=torch.int32, device="cuda")
    with pytest.raises(binding.GmError) as e:
        binding.gm_row_ptr_shift(rp32, 20)
    assert e.value.status == 3  # GM_ERR_INDEX_OVERFLOW, nothing changed
    assert rp32.tolist() == [0, 5, 2 ** 31 - 10]
    binding.gm_row_ptr_shift(rp32, 9)
    assert rp32.tolist() == [9, 14, 2 ** 31 - 1]
