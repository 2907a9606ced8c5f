"""The allocation-free prefix sum (gm_prefix_sum_noalloc) against the existing path.

Some callers cannot allocate device memory while they run (work captured into a
CUDA graph, callbacks and real-time loops that must not block on an allocator,
hosts whose framework owns all device memory). gm_prefix_sum_noalloc gives them
the scan that places C.rowPtr, with its scratch in a fixed array of the library.
This test calls it through the C ABI twice in a row, on the row counts of two
different products, and checks each result against the C.rowPtr that
gm_spgemm_symbolic produced for the same product. The values are integers, so
the comparison is exact.
"""
import ctypes

import numpy as np
import pytest

from sparse_gemm_irregular_gm_gb300 import binding, inputs as gi

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return binding.load()


def _symbolic_row_ptr(A):
    """C.rowPtr of A @ A from the existing path (analyze + symbolic)."""
    Ad = binding.to_device(A)
    plan = binding.gm_spgemm_analyze(Ad, Ad)
    try:
        rp = torch.empty(A.n_rows + 1, dtype=torch.int64, device="cuda")
        nnz = binding.gm_spgemm_symbolic(plan, rp)
    finally:
        binding.gm_spgemm_plan_destroy(plan)
    return rp, nnz


def test_noalloc_scan_matches_symbolic_row_ptr_twice(lib):
    stream = torch.cuda.current_stream()
    for A in (gi.rmat(12, 8, seed=3), gi.laplacian_2d(300, 200)):  # two calls in a row
        rp, nnz = _symbolic_row_ptr(A)
        counts = (rp[1:] - rp[:-1]).contiguous()          # row nnz of C
        out = torch.full_like(counts, -1)
        total = torch.full((1,), -1, dtype=torch.int64, device="cuda")
        rc = lib.gm_prefix_sum_noalloc(ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                       counts.numel(), ctypes.c_void_p(total.data_ptr()),
                                       ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, binding.gm_status_string(rc)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), rp[:-1].cpu().numpy())
        assert int(total.item()) == nnz == int(rp[-1])


def test_noalloc_scan_in_place_and_multilevel(lib):
    # more than 2048 * 2048 elements: two levels of partial sums in the fixed array
    n = 5_000_000
    x = torch.randint(0, 7, (n,), dtype=torch.int64, device="cuda")
    ref = torch.cumsum(x, 0) - x
    binding.gm_prefix_sum_noalloc(x, x)  # in place
    torch.cuda.synchronize()
    assert torch.equal(x, ref)


def test_noalloc_scan_rejects_oversize_and_bad_args(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: both calls fail before any launch
    assert lib.gm_prefix_sum_noalloc(fake, fake, (1 << 27) + 1, None, None) == 5  # GM_ERR_WORKSPACE
    assert lib.gm_prefix_sum_noalloc(None, None, 10, None, None) == 1             # GM_ERR_INVALID_ARG
    assert lib.gm_prefix_sum_noalloc(None, None, 0, None, None) == 0              # empty: nothing to do
