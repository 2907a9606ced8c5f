"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle (structure bit-exact, fp64 values within
1e-12 * sum|a_ik * b_kj| per entry)."""
import numpy as np

import oracle
from sparse_gemm_irregular_gm_gb300 import binding

REL_TOL = 1e-12


F32_EPS = 2.0 ** -24  # unit roundoff of float


def run_gpu(A, B, return_info=False, dtype=None, **cfg):
    import torch
    Ad, Bd = binding.to_device(A, dtype=dtype), binding.to_device(B, dtype=dtype)
    C, info = binding.spgemm(Ad, Bd, binding.make_config(**cfg) if cfg else None, return_info=True)
    torch.cuda.synchronize()
    out = (C.row_ptr.cpu().numpy(), C.col.cpu().numpy(), C.val.cpu().numpy())
    return (out, info) if return_info else out


def assert_matches(ref, rp, col, val, exact=False):
    """ref: oracle.OracleC over the same rows (in order); rp/col/val: GPU rows."""
    np.testing.assert_array_equal(np.diff(rp), np.diff(ref.row_ptr), err_msg="row nnz differ")
    np.testing.assert_array_equal(col, ref.col, err_msg="columns differ")
    if exact:
        np.testing.assert_array_equal(val, ref.val, err_msg="integer-valued results differ")
    else:
        err = np.abs(val - ref.val)
        bound = REL_TOL * ref.abs_scale
        bad = np.nonzero(err > bound)[0]
        assert bad.size == 0, f"{bad.size} values outside 1e-12*sum|ab|; worst rel {np.max(err / np.maximum(ref.abs_scale, 1e-300))}"


def check_full(A, B, exact=False, **cfg):
    (rp, col, val), info = run_gpu(A, B, return_info=True, **cfg)
    ref = oracle.spgemm(A, B)
    assert rp[0] == 0
    assert_matches(ref, rp, col, val, exact)
    return info


def gather_rows(C, rows):
    """Host copies of the given rows of a device CSR result."""
    import torch
    rp = C.row_ptr.cpu().numpy().astype(np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    lo, hi = rp[rows], rp[rows + 1]
    lens = hi - lo
    srp = np.zeros(len(rows) + 1, dtype=np.int64)
    np.cumsum(lens, out=srp[1:])
    idx = np.repeat(lo - srp[:-1], lens) + np.arange(srp[-1], dtype=np.int64)  # entry positions in C
    t = torch.from_numpy(idx).to(C.col.device)
    col = C.col[t].cpu().numpy()
    val = C.val[t].cpu().numpy()
    return srp, col, val


def check_invariants(C, u):
    """Properties every result must have, checked on the device in slices."""
    import torch
    rp = C.row_ptr
    n = rp.numel() - 1
    assert int(rp[0]) == 0 and int(rp[-1]) == C.col.numel()
    lens = rp[1:] - rp[:-1]
    assert bool((lens >= 0).all())
    assert bool((lens.cpu() <= torch.from_numpy(u)).all()), "a row has more entries than products"
    nnz = C.col.numel()
    start = torch.zeros(1, dtype=torch.bool, device=rp.device)
    step = 1 << 28
    rp_cpu = rp.cpu().numpy()
    for lo in range(0, nnz, step):
        hi = min(nnz, lo + step + 1)
        c = C.col[lo:hi].to(torch.int64)
        first = torch.zeros(hi - lo, dtype=torch.bool, device=rp.device)
        s = rp_cpu[(rp_cpu >= lo) & (rp_cpu < hi)] - lo
        first[torch.from_numpy(s).to(rp.device)] = True
        ok = (c[1:] > c[:-1]) | first[1:]
        assert bool(ok.all()), "columns not strictly increasing within a row"
        assert int(c.min()) >= 0 and int(c.max()) < C.n_cols
    del start
    return n


def rounded_to_f32(M):
    """M with its values rounded to float (and held as float64, for the oracle)."""
    return M.__class__(M.n_rows, M.n_cols, M.row_ptr, M.col, M.val.astype(np.float32).astype(np.float64))


def ones_like_csr(M):
    return M.__class__(M.n_rows, M.n_cols, M.row_ptr, M.col, np.ones_like(M.val))


def assert_matches_f32(ref, ref_k, rp, col, val):
    """Float results against the oracle over the same float inputs: structure
    bit-exact, every entry within 2 k u sum|ab| (k from ref_k, the oracle on
    all-ones values)."""
    np.testing.assert_array_equal(np.diff(rp), np.diff(ref.row_ptr), err_msg="row nnz differ")
    np.testing.assert_array_equal(col, ref.col, err_msg="columns differ")
    err = np.abs(val.astype(np.float64) - ref.val)
    bad = np.nonzero(err > 2.0 * ref_k.val * F32_EPS * ref.abs_scale)[0]
    assert bad.size == 0, f"{bad.size} float values outside 2 k u sum|ab|"


def check_full_f32(A, B, exact=False, **cfg):
    """C = A*B with float values (gm_config.value_type = GM_VALUE_F32). The inputs
    are rounded to float first and the oracle sums the same float values in fp64.
    Structure bit-exact; integer-valued inputs exactly; otherwise every entry
    within 2 k u sum|a_ik b_kj|, u = 2^-24 and k = the entry's number of products
    (the oracle's value on all-ones inputs): a float product is within u of the
    exact one and a sum of k terms in any order within (k - 1) u of the exact sum,
    relative to the sum of the magnitudes."""
    A32, B32 = rounded_to_f32(A), rounded_to_f32(B)
    (rp, col, val), info = run_gpu(A32, B32, return_info=True, dtype=np.float32, **cfg)
    assert val.dtype == np.float32 and info.value_type == binding.GM_VALUE_F32
    ref = oracle.spgemm(A32, B32)
    np.testing.assert_array_equal(np.diff(rp), np.diff(ref.row_ptr), err_msg="row nnz differ")
    np.testing.assert_array_equal(col, ref.col, err_msg="columns differ")
    v = val.astype(np.float64)
    if exact:
        np.testing.assert_array_equal(v, ref.val, err_msg="integer-valued float results differ")
    else:
        k = oracle.spgemm(ones_like_csr(A), ones_like_csr(B)).val
        bound = 2.0 * k * F32_EPS * ref.abs_scale
        err = np.abs(v - ref.val)
        bad = np.nonzero(err > bound)[0]
        assert bad.size == 0, f"{bad.size} float values outside 2 k u sum|ab|"
    return info
