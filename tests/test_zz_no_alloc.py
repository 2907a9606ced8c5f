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


@pytest.mark.parametrize("n", [1, 2047, 2048, 2049, 2048 * 3000, 2048 * 2048, 2048 * 2048 + 1])
def test_noalloc_scan_at_tile_edges(lib, n):
    """Sizes on and next to the edges of the 2048-element tiles and of the first
    level of partial sums (2048 tiles), against torch.cumsum."""
    x = torch.randint(0, 1000, (n,), dtype=torch.int64, device="cuda")
    out = torch.empty_like(x)
    total = torch.empty(1, dtype=torch.int64, device="cuda")
    binding.gm_prefix_sum_noalloc(x, out, total)
    torch.cuda.synchronize()
    ref = torch.cumsum(x, 0)
    assert torch.equal(out, ref - x) and int(total.item()) == int(ref[-1])


def test_noalloc_scan_at_the_largest_size(lib):
    """n = 2^27, the largest size the fixed array serves: 65,536 tiles fill the
    first level of partial sums exactly. In place (1 GiB), against torch.cumsum."""
    n = 1 << 27
    x = torch.randint(0, 1 << 20, (n,), dtype=torch.int64, device="cuda")
    ref = torch.cumsum(x, 0)
    total = torch.empty(1, dtype=torch.int64, device="cuda")
    binding.gm_prefix_sum_noalloc(x, x, total)
    torch.cuda.synchronize()
    assert int(total.item()) == int(ref[-1])
    assert torch.equal(x[1:], ref[:-1]) and int(x[0]) == 0  # exclusive: out[i] = inclusive[i - 1]
    del x, ref


def test_noalloc_binding_rejects_bad_tensors(lib):
    x = torch.zeros(100, dtype=torch.int64, device="cuda")
    with pytest.raises(ValueError):
        binding.gm_prefix_sum_noalloc(x, torch.zeros(99, dtype=torch.int64, device="cuda"))
    with pytest.raises(ValueError):
        binding.gm_prefix_sum_noalloc(x, torch.zeros(100, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        binding.gm_prefix_sum_noalloc(x, torch.zeros(200, dtype=torch.int64, device="cuda")[::2])
    with pytest.raises(ValueError):
        binding.gm_prefix_sum_noalloc(x.cpu(), x)
    with pytest.raises(ValueError):
        binding.gm_prefix_sum_noalloc(x, x, torch.zeros(0, dtype=torch.int64, device="cuda"))


def _library_cudart():
    """The CUDA runtime the library is linked to (the libcudart.so.* mapped in this
    process; loading it again by path returns the same instance)."""
    with open("/proc/self/maps") as f:
        paths = [ln.split()[-1] for ln in f if "/libcudart.so" in ln]
    return ctypes.CDLL(paths[0] if paths else "libcudart.so.13")


def test_noalloc_leaves_an_earlier_error_pending(lib):
    """A CUDA error that earlier work left pending is reported (GM_ERR_CUDA), is
    not cleared, and nothing is queued; once its owner has read it, the next call
    works. The earlier error is the runtime's host-side refusal of a device
    ordinal that does not exist (no GPU work is involved)."""
    cudart = _library_cudart()
    x = torch.arange(10, dtype=torch.int64, device="cuda")
    out = torch.full_like(x, -1)
    torch.cuda.synchronize()
    cudart.cudaGetLastError()
    count = ctypes.c_int(0)
    assert cudart.cudaGetDeviceCount(ctypes.byref(count)) == 0
    # No torch call between here and the read below: torch checks (and clears)
    # the pending error after its own launches.
    assert cudart.cudaSetDevice(count.value + 7) != 0  # invalid ordinal: refused on the host
    rc = lib.gm_prefix_sum_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()), 10, None,
                                   None)
    assert rc == 6  # GM_ERR_CUDA
    assert cudart.cudaGetLastError() != 0  # still pending for its owner, now read and cleared
    torch.cuda.synchronize()
    assert int(out[0]) == -1  # nothing was queued
    binding.gm_prefix_sum_noalloc(x, out)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.cumsum(x, 0) - x)


def test_noalloc_scan_rejects_oversize_and_bad_args(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: both calls fail before any launch
    assert lib.gm_prefix_sum_noalloc(fake, fake, (1 << 27) + 1, None, None) == 5  # GM_ERR_WORKSPACE
    assert lib.gm_prefix_sum_noalloc(None, None, 10, None, None) == 1             # GM_ERR_INVALID_ARG
    assert lib.gm_prefix_sum_noalloc(None, None, 0, None, None) == 0              # empty: nothing to do
