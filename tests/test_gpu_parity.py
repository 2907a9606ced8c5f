"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Structure (row pointers, columns, nnz) must match bit for bit; fp64 values
within 1e-12 * sum|a_ik * b_kj| per entry; integer-valued inputs exactly.
Small inputs force every path (heavy rows, one and several multisplit levels,
no level, several workspace batches, both pipelines); the five workloads run
at their full sizes: R-MAT scale 18 is compared row by row in full, scale 20
on 50,000 rows stratified by their products plus invariants on every row (in
full with GM_FULL_PARITY_20=1).
"""
import json
import os

import numpy as np
import pytest

import oracle
from sparse_gemm_irregular_gm_gb300 import binding, inputs as gi
from tests.gpu_common import (assert_matches, assert_matches_f32, check_full, check_full_f32, check_invariants,
                               gather_rows, ones_like_csr, rounded_to_f32, run_gpu)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


# forced paths on small inputs: (name, config)
FORCED = [
    ("auto", {}),
    ("heavy_L0", {"tau": 16}),                                          # C.m <= D: no multisplit
    ("heavy_L1", {"tau": 16, "dense_width": 128, "n_chunks_max": 16}),  # one level, 8 chunks
    ("heavy_L2", {"tau": 16, "dense_width": 64, "n_chunks_max": 4}),    # two levels
    ("heavy_L3", {"tau": 16, "dense_width": 16, "n_chunks_max": 4}),    # three levels
    ("unfused", {"tau": 16, "dense_width": 64, "n_chunks_max": 4, "pipeline": binding.GM_PIPE_UNFUSED}),
    ("batched", {"tau": 16, "dense_width": 128, "n_chunks_max": 16, "workspace_cap_bytes": 6 << 20,
                 "pipeline": binding.GM_PIPE_FUSED_HISTO}),
    ("L1_unfused", {"tau": 16, "dense_width": 128, "n_chunks_max": 16, "pipeline": binding.GM_PIPE_UNFUSED}),
    ("L1_wide_chunks", {"tau": 64, "dense_width": 512}),                   # one level, 2 chunks of 512
    ("L1_outer", {"tau": 16, "dense_width": 128, "n_chunks_max": 16, "pipeline": binding.GM_PIPE_FUSED_HISTO}),
    ("L1_rowwise_batched", {"tau": 16, "dense_width": 128, "n_chunks_max": 16, "workspace_cap_bytes": 5 << 20,
                            "pipeline": binding.GM_PIPE_ROWWISE}),
    ("L1_rowwise", {"tau": 16, "dense_width": 128, "n_chunks_max": 16, "pipeline": binding.GM_PIPE_ROWWISE}),
    ("L2_outer", {"tau": 16, "dense_width": 64, "n_chunks_max": 4, "pipeline": binding.GM_PIPE_FUSED_HISTO}),
    ("L3_outer", {"tau": 16, "dense_width": 16, "n_chunks_max": 4, "pipeline": binding.GM_PIPE_FUSED_HISTO}),
    ("L1_rowwise_256", {"tau": 16, "dense_width": 256, "n_chunks_max": 16, "pipeline": binding.GM_PIPE_ROWWISE}),
]


@pytest.mark.parametrize("name,cfg", FORCED, ids=[f[0] for f in FORCED])
@pytest.mark.parametrize("values", ["uniform", "int"])
def test_rmat10_forced_paths(name, cfg, values):
    A = gi.rmat(10, 8, seed=1, values=values)
    info = check_full(A, A, exact=values == "int", **cfg)
    if name != "auto":
        assert info.n_heavy_rows > 0
        if "batched" in name:
            assert info.n_batches > 1
        if name in ("heavy_L1", "L1_wide_chunks", "L1_rowwise_batched", "L1_rowwise"):
            assert info.pipeline == binding.GM_PIPE_ROWWISE
        if name == "L1_rowwise_256":
            assert info.pipeline == binding.GM_PIPE_ROWWISE
        if name in ("heavy_L2", "heavy_L3"):  # level 0 by the row-order expansion
            assert info.pipeline == binding.GM_PIPE_ROWWISE and info.params.n_levels >= 2
        if name in ("L2_outer", "L3_outer"):
            assert info.pipeline == binding.GM_PIPE_FUSED_HISTO and info.params.n_levels >= 2
        if name == "L1_outer":
            assert info.pipeline == binding.GM_PIPE_FUSED_HISTO


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("shape", [(33, 20, 41), (64, 64, 64), (200, 90, 300), (1, 50, 7), (70, 1, 70)])
@pytest.mark.parametrize("cfg", [{}, {"tau": 2, "dense_width": 4, "n_chunks_max": 2}], ids=["auto", "forced"])
def test_random_irregular(seed, shape, cfg):
    m, k, n = shape
    A = gi.random_csr(m, k, 0.3, seed, values="int", unsorted=True, duplicates=True, explicit_zeros=True,
                      empty_rows=0.2)
    B = gi.random_csr(k, n, 0.3, seed + 50, values="int", unsorted=True, duplicates=True, explicit_zeros=True,
                      empty_rows=0.2)
    check_full(A, B, exact=True, **cfg)


@pytest.mark.parametrize("scale", [11, 12])
def test_symbolic_paths_agree(scale):
    """Whole-row bitmap symbolic (default) and the C-hat_reord symbolic give the same C."""
    A = gi.rmat(scale, 16, seed=scale)
    cfg = {"tau": 256, "dense_width": 256, "n_chunks_max": 16}
    r1 = run_gpu(A, A, **cfg)
    r2 = run_gpu(A, A, pipeline=binding.GM_PIPE_UNFUSED, **cfg)
    np.testing.assert_array_equal(r1[0], r2[0])
    np.testing.assert_array_equal(r1[1], r2[1])
    ref = oracle.spgemm(A, A)
    assert_matches(ref, *r1)


def test_empty_and_degenerate():
    empty = gi.random_csr(8, 6, 0.0, 1)
    B = gi.random_csr(6, 9, 0.5, 2)
    (rp, col, val) = run_gpu(empty, B)
    assert rp.tolist() == [0] * 9 and col.size == 0
    (rp, col, val) = run_gpu(B.__class__(6, 6, np.zeros(7, np.int64), np.zeros(0, np.int32), np.zeros(0)), B)
    assert col.size == 0
    one = gi.identity(1)
    (rp, col, val) = run_gpu(one, one)
    assert rp.tolist() == [0, 1] and col.tolist() == [0] and val.tolist() == [1.0]
    zero_rows = gi.CSR(0, 5, np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0))
    (rp, col, val) = run_gpu(zero_rows, gi.random_csr(5, 4, 0.5, 3))
    assert rp.tolist() == [0] and col.size == 0
    # one dense row against a dense block: a single heavy row
    A = gi.random_csr(3, 300, 1.0, 4, values="int")
    Bd = gi.random_csr(300, 500, 0.9, 5, values="int")
    check_full(A, Bd, exact=True, tau=100, dense_width=128, n_chunks_max=4)


def test_bad_index_and_bad_row_ptr_are_reported():
    A = gi.random_csr(10, 10, 0.4, 1)
    bad = gi.CSR(A.n_rows, A.n_cols, A.row_ptr.copy(), A.col.copy(), A.val.copy())
    bad.col[3] = 10  # == n_cols: out of range
    with pytest.raises(binding.GmError) as e:
        binding.spgemm(binding.to_device(bad), binding.to_device(A))
    assert e.value.status == 9
    bad2 = gi.CSR(A.n_rows, A.n_cols, A.row_ptr.copy(), A.col.copy(), A.val.copy())
    bad2.row_ptr[4], bad2.row_ptr[5] = bad2.row_ptr[5] + 1, bad2.row_ptr[4]
    with pytest.raises(binding.GmError) as e:
        binding.spgemm(binding.to_device(A), binding.to_device(bad2))
    assert e.value.status == 9


def test_call_order_is_enforced():
    A = gi.random_csr(10, 10, 0.4, 1)
    Ad = binding.to_device(A)
    plan = binding.gm_spgemm_analyze(Ad, Ad)
    try:
        c = torch.empty(0, dtype=torch.int32, device="cuda")
        v = torch.empty(0, dtype=torch.float64, device="cuda")
        with pytest.raises(binding.GmError) as e:
            binding.gm_spgemm_numeric(plan, c, v)
        assert e.value.status == 8
        rp = torch.empty(11, dtype=torch.int64, device="cuda")
        nnz = binding.gm_spgemm_symbolic(plan, rp)
        with pytest.raises(binding.GmError) as e:
            binding.gm_spgemm_symbolic(plan, rp)
        assert e.value.status == 8
        binding.gm_spgemm_numeric(plan, torch.empty(nnz, dtype=torch.int32, device="cuda"),
                                  torch.empty(nnz, dtype=torch.float64, device="cuda"))
    finally:
        binding.gm_spgemm_plan_destroy(plan)


# --- stage parity through the debug views -----------------------------------------

def _analyze_keep(A, B, **cfg):
    Ad, Bd = binding.to_device(A), binding.to_device(B)
    cfg["flags"] = cfg.get("flags", 0) | binding.GM_FLAG_KEEP_INTERMEDIATES
    plan = binding.gm_spgemm_analyze(Ad, Bd, binding.make_config(**cfg))
    return plan, (Ad, Bd)


def test_stage1_counts_partition_and_chat_rowptr():
    A = gi.rmat(10, 8, seed=2)
    tau = 300
    plan, keep = _analyze_keep(A, A, tau=tau)
    try:
        u = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_IP_COUNTS)
        np.testing.assert_array_equal(u, oracle.ip_counts(A, A))
        heavy, light = oracle.thresh_partition(u, tau)
        np.testing.assert_array_equal(binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_HEAVY_ROWS), heavy)
        np.testing.assert_array_equal(np.sort(binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_LIGHT_ROWS)), light)
        rp = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_CHAT_ROWPTR)
        np.testing.assert_array_equal(np.diff(rp), u[heavy])
        assert rp[0] == 0
    finally:
        binding.gm_spgemm_plan_destroy(plan)


def test_heavy_threshold_is_strict():
    """A row whose intermediate products equal tau exactly is light: heavy means
    exceeding tau (gMAGNUS Sec. I, Sec. II-B). tau is set to a product count that
    occurs; the partition is checked against the oracle's ThreshPartition and the
    product against the oracle."""
    A = gi.rmat(10, 8, seed=2)
    u = oracle.ip_counts(A, A)
    cand = np.unique(u[(u >= 64) & (u <= 2000)])
    tau = int(cand[len(cand) // 2])
    assert (u == tau).any()
    ref_heavy, ref_light = oracle.thresh_partition(u, tau)
    plan, keep = _analyze_keep(A, A, tau=tau)
    try:
        heavy = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_HEAVY_ROWS)
        np.testing.assert_array_equal(heavy, ref_heavy)
        assert np.isin(np.nonzero(u == tau)[0], ref_light).all()
    finally:
        binding.gm_spgemm_plan_destroy(plan)
    info = check_full(A, A, tau=tau)
    assert info.n_heavy_rows == int((u > tau).sum()) > 0


def _run_symbolic(plan, n_rows):
    rp = torch.empty(n_rows + 1, dtype=torch.int64, device="cuda")
    return binding.gm_spgemm_symbolic(plan, rp)


def _multiset(cols, vals):
    return sorted(zip(cols.tolist(), np.round(vals, 12).tolist()))


@pytest.mark.parametrize("cfg", [{"tau": 16, "dense_width": 64, "n_chunks_max": 4},
                                 {"tau": 16, "dense_width": 128, "n_chunks_max": 16},
                                 {"tau": 16, "dense_width": 16, "n_chunks_max": 4,
                                  "pipeline": binding.GM_PIPE_UNFUSED}])
def test_outer_product_and_multisplit_levels(cfg):
    A = gi.rmat(9, 8, seed=4, values="int")
    plan, keep = _analyze_keep(A, A, **cfg)
    try:
        _run_symbolic(plan, A.n_rows)
        params = binding.gm_spgemm_plan_info(plan).params
        heavy = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_HEAVY_ROWS)
        rp = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_CHAT_ROWPTR)
        col = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_CHAT_COL)
        val = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_CHAT_VAL)
        ref = oracle.expand_rows(A, A, heavy)
        for h, items in enumerate(ref):  # C-hat rows as multisets (Fig. 1, outer product)
            got = _multiset(col[rp[h]:rp[h + 1]], val[rp[h]:rp[h + 1]])
            assert got == sorted((c, round(v, 12)) for c, v in items)
        # each level: chunk c of parent p holds the parent's elements in its column range
        parents = [sorted((c, round(v, 12)) for c, v in items) for items in ref]
        for lev in range(params.n_levels):
            v, w = params.v_chunks[lev], params.widths[lev]
            rrp = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_REORD_ROWPTR, lev)
            rcol = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_REORD_COL, lev)
            rval = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_REORD_VAL, lev)
            child = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_REORD_CHILD, lev)
            expect = {}
            for pi, items in enumerate(parents):
                for ci, ch in enumerate(oracle.split_chunks(items, v, w)):
                    expect[pi * v + ci] = sorted(ch)
            assert len(child) == len(expect)
            for m, ch in enumerate(child):
                assert _multiset(rcol[rrp[m]:rrp[m + 1]], rval[rrp[m]:rrp[m + 1]]) == expect[int(ch)]
            # heavy chunks first, in order; they are the next level's parents
            counts = np.diff(rrp)
            nh = int((counts > params.tau).sum()) if lev < params.n_levels - 1 else 0
            if lev < params.n_levels - 1:
                assert np.all(counts[:nh] > params.tau) and np.all(counts[nh:] <= params.tau)
                assert np.all(np.diff(child[:nh]) > 0)
            parents = [expect[int(ch)] for ch in child[:nh]]
    finally:
        binding.gm_spgemm_plan_destroy(plan)


def test_fig1_worked_example_on_gpu():
    with open(os.path.join(GOLDEN, "fig1_worked_example.json")) as f:
        g = json.load(f)
    rng = np.random.default_rng(7)
    syms = {}

    def sym(s):
        return syms.setdefault(s, float(rng.integers(2, 40)))

    def build(rows, shape):
        rp, col, val = [0], [], []
        for i in range(shape[0]):
            for c, s in rows.get(str(i), []):
                col.append(c)
                val.append(sym(s))
            rp.append(len(col))
        return gi.CSR(shape[0], shape[1], np.array(rp, np.int64), np.array(col, np.int32), np.array(val))

    A, B = build(g["A_rows"], g["A_shape"]), build(g["B_rows"], g["B_shape"])
    plan, keep = _analyze_keep(A, B, tau=2, dense_width=4, n_chunks_max=2)
    try:
        _run_symbolic(plan, A.n_rows)
        assert binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_HEAVY_ROWS).tolist() == g["heavy_rows"]
        rp = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_CHAT_ROWPTR)
        col = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_CHAT_COL)
        for h, cols in enumerate(g["Chat_col"]):
            assert sorted(col[rp[h]:rp[h + 1]].tolist()) == sorted(cols)
        rrp = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_REORD_ROWPTR, 0)
        rcol = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_REORD_COL, 0)
        for k, cols in enumerate(g["Creord_col"]):
            assert sorted(rcol[rrp[k]:rrp[k + 1]].tolist()) == sorted(cols)
    finally:
        binding.gm_spgemm_plan_destroy(plan)
    prod = lambda s: sym(s[:3]) * sym(s[3:])
    (crp, ccol, cval) = run_gpu(A, B, tau=2, dense_width=4, n_chunks_max=2)
    for r, entries in g["C_rows"].items():
        i = int(r)
        assert ccol[crp[i]:crp[i + 1]].tolist() == [c for c, _ in entries]
        assert cval[crp[i]:crp[i + 1]].tolist() == [sum(prod(s) for s in labels) for _, labels in entries]


def _light_rows_case(n_cols, seed):
    """A with rows whose products fill every light bin (u from 1 to tau) and one
    heavy row, some with thousands of A entries (several entry tiles of the
    light-row kernels) and with empty B rows among the selected ones; B rows of
    length 0, 1, 2 and a few long ones (1500). Integer values."""
    rng = np.random.default_rng(seed)
    nb = 12000
    lens = np.ones(nb, np.int64)
    lens[::7] = 2
    lens[5::97] = 0
    lens[:6] = 1500
    b_rp = np.zeros(nb + 1, np.int64)
    np.cumsum(lens, out=b_rp[1:])
    b_col = np.concatenate([np.sort(rng.choice(n_cols, int(l), replace=False)) for l in lens]).astype(np.int32)
    B = gi.CSR(nb, n_cols, b_rp, b_col, rng.integers(-3, 4, b_col.size).astype(np.float64))
    rows = []
    for target in (1, 17, 40, 100, 200, 500, 1000, 1500, 3000, 5000, 7000, 7900, 8450, 9686):
        cols = list(rng.choice(np.arange(6, nb), min(target, nb - 6), replace=False))
        rows.append(cols)
    rows.append([0, 1, 2, 3, 4] + list(rng.choice(np.arange(6, nb), 40, replace=False)))  # long B rows
    rows.append(list(range(5, nb, 97))[:50] + [6, 7, 8])  # mostly empty B rows
    a_rp = np.zeros(len(rows) + 1, np.int64)
    np.cumsum([len(r) for r in rows], out=a_rp[1:])
    a_col = np.concatenate([np.sort(np.asarray(r)) for r in rows]).astype(np.int32)
    A = gi.CSR(len(rows), nb, a_rp, a_col, rng.integers(-3, 4, a_col.size).astype(np.float64))
    return A, B


@pytest.mark.parametrize("n_cols", [1 << 20, 3000])
def test_light_rows_every_bin_and_entry_tiles(n_cols):
    A, B = _light_rows_case(n_cols, seed=n_cols % 97)
    u = oracle.ip_counts(A, B)
    assert u.max() > 9685 and ((u > 1024) & (u <= 9685)).sum() >= 5
    info = check_full(A, B, exact=True)
    assert info.n_heavy_rows == int((u > info.params.tau).sum())


@pytest.mark.parametrize("values", ["uniform", "int"])
def test_rowwise_sorted_and_unsorted_b(values):
    """The row-order pipeline scatters whole runs of a B row into a chunk when B's
    rows are sorted, and product by product otherwise: both give the oracle's C."""
    A = gi.rmat(11, 8, seed=5, values=values)
    rng = np.random.default_rng(7)
    perm = np.concatenate([lo + rng.permutation(hi - lo) for lo, hi in zip(A.row_ptr[:-1], A.row_ptr[1:])])
    B_unsorted = gi.CSR(A.n_rows, A.n_cols, A.row_ptr.copy(), A.col[perm].copy(), A.val[perm].copy())
    cfg = {"tau": 16, "dense_width": 128, "n_chunks_max": 16, "pipeline": binding.GM_PIPE_ROWWISE}
    for B in (A, B_unsorted):
        info = check_full(A, B, exact=values == "int", **cfg)
        assert info.pipeline == binding.GM_PIPE_ROWWISE and info.n_heavy_rows > 0


def _rows_of(M, rows):
    rows = np.asarray(rows, dtype=np.int64)
    lens = M.row_ptr[rows + 1] - M.row_ptr[rows]
    rp = np.zeros(rows.size + 1, np.int64)
    np.cumsum(lens, out=rp[1:])
    idx = np.concatenate([np.arange(M.row_ptr[r], M.row_ptr[r + 1]) for r in rows])
    return gi.CSR(rows.size, M.n_cols, rp, M.col[idx].copy(), M.val[idx].copy())


@pytest.mark.parametrize("pipeline", [binding.GM_PIPE_FUSED_HISTO, binding.GM_PIPE_AUTO], ids=["outer", "auto"])
def test_large_chunks_many_tiles_exact(pipeline):
    """The heaviest rows of a scale-16 R-MAT times the whole matrix: chunks of
    tens of thousands of elements (many tiles of the large-chunk accumulators)
    with the R-MAT's hot columns; integer values, so exact."""
    A = gi.rmat(16, 16, seed=3, values="int")
    u = oracle.ip_counts(A, A)
    rows = np.concatenate([np.argsort(u)[-40:], np.random.default_rng(0).choice(A.n_rows, 40, replace=False)])
    As = _rows_of(A, rows)
    info = check_full(As, A, exact=True, pipeline=pipeline)
    assert info.n_heavy_rows >= 40 and u[rows].max() > 16 * 4096
    # some chunks have more than 8192 columns: with double values the streamed
    # accumulator (bulk copies into shared memory) takes them in the row-order pipeline
    ref = oracle.spgemm(As, A)
    widest = max(np.bincount(ref.col[ref.row_ptr[i]:ref.row_ptr[i + 1]] >> 14).max() for i in range(As.n_rows)
                 if ref.row_ptr[i + 1] > ref.row_ptr[i])
    assert widest > 8192
    assert info.pipeline == (binding.GM_PIPE_ROWWISE if pipeline == binding.GM_PIPE_AUTO else pipeline)


@pytest.mark.parametrize("pipeline", [binding.GM_PIPE_FUSED_HISTO, binding.GM_PIPE_AUTO], ids=["outer", "auto"])
@pytest.mark.parametrize("n_hot", [5000, 13000])
def test_chunk_with_one_hot_column(n_hot, pipeline):
    """A chunk whose elements nearly all fall on one column: one run of equal rank
    crosses every thread of every tile. Row 0: n_hot products on column 7; row 1:
    the same plus products spread over the chunk; integer values."""
    rng = np.random.default_rng(n_hot)
    n_cols = 40000  # 4 chunks of 16384 at the default dense width
    nb = n_hot + 3000
    b_lens = np.ones(nb, np.int64)
    b_lens[n_hot:] = 3
    b_rp = np.zeros(nb + 1, np.int64)
    np.cumsum(b_lens, out=b_rp[1:])
    b_col = np.full(int(b_rp[-1]), 7, np.int32)
    tail = b_col[b_rp[n_hot]:]
    tail[:] = rng.integers(0, n_cols, tail.size).astype(np.int32)
    for k in range(n_hot, nb):  # distinct columns inside each B row
        seg = b_col[b_rp[k]:b_rp[k + 1]]
        seg[:] = np.sort(rng.choice(n_cols, seg.size, replace=False))
    B = gi.CSR(nb, n_cols, b_rp, b_col, rng.integers(-3, 4, b_col.size).astype(np.float64))
    r0 = np.arange(n_hot)
    r1 = np.arange(nb)
    a_col = np.concatenate([r0, r1]).astype(np.int32)
    A = gi.CSR(2, nb, np.array([0, r0.size, r0.size + r1.size], np.int64), a_col,
               rng.integers(1, 4, a_col.size).astype(np.float64))
    info = check_full(A, B, exact=True, tau=64, pipeline=pipeline)
    assert info.pipeline == (binding.GM_PIPE_ROWWISE if pipeline == binding.GM_PIPE_AUTO else pipeline)


@pytest.mark.parametrize("pipeline", [binding.GM_PIPE_AUTO, binding.GM_PIPE_FUSED_HISTO], ids=["rowexp", "outer"])
@pytest.mark.parametrize("values", ["uniform", "int"])
def test_multilevel_wide_light_chunks(values, pipeline):
    """Three levels (4, 4, 2 chunks of 4096, 1024, 512 columns) with tau = 2048:
    about 8900 level-0 chunks of 513-2048 elements leave the hierarchy as light
    chunks, summed by the bitmap-rank accumulator at width 4096; level 0 from the
    row-order expansion or from C-hat."""
    A = gi.rmat(14, 16, seed=4, values=values)
    info = check_full(A, A, exact=values == "int", tau=2048, dense_width=512, n_chunks_max=4, pipeline=pipeline)
    assert info.params.n_levels == 3 and info.n_heavy_rows > 4000
    assert info.pipeline == (binding.GM_PIPE_ROWWISE if pipeline == binding.GM_PIPE_AUTO else pipeline)


@pytest.mark.parametrize("values", ["uniform", "int"])
def test_sorted_b_rows_that_repeat_a_column(values):
    """B rows sorted but repeating a column: the row-order expansion still writes
    each run of a B row into its chunk contiguously, and the repeated column's
    products add. Both the plain and the repeating B give the oracle's C."""
    A = gi.rmat(11, 8, seed=5, values=values)
    rp, col, val = A.row_ptr, A.col, A.val
    rows = [r for r in range(A.n_rows) if rp[r + 1] - rp[r] >= 2][:50]
    col2 = np.insert(col, rp[rows], col[rp[rows]])  # each chosen row starts with its first column twice
    val2 = np.insert(val, rp[rows], val[rp[rows]])
    rp2 = rp + np.searchsorted(np.asarray(rows), np.arange(A.n_rows + 1), side="left")
    B_dup = gi.CSR(A.n_rows, A.n_cols, rp2.astype(np.int64), col2.astype(np.int32), val2)
    B_dup.check()
    assert np.all(np.diff(B_dup.col[B_dup.row_ptr[rows[0]]:B_dup.row_ptr[rows[0] + 1]]) >= 0)
    cfg = {"tau": 16, "dense_width": 128, "n_chunks_max": 16}
    info = check_full(A, A, exact=values == "int", **cfg)
    assert info.pipeline == binding.GM_PIPE_ROWWISE
    info = check_full(A, B_dup, exact=values == "int", **cfg)
    assert info.pipeline == binding.GM_PIPE_ROWWISE and info.n_heavy_rows > 0


@pytest.mark.parametrize("a_density", [4, 16])
def test_rmat_grid_pairs(a_density):
    """A*B with independent R-MAT A and B (the pages' grid: A.nnz/A.n varied, B.nnz/B.n
    = 8) at scale 13; statistics of the kind Table III reports checked against the
    oracle's own counts."""
    A, B = gi.named_pair(f"rmatAB_s13_a{a_density}_b8", seed=2)
    u = oracle.ip_counts(A, B)
    info = check_full(A, B)
    assert info.ip_total == int(u.sum()) and info.n_heavy_rows == int((u > info.params.tau).sum())


# --- float values (gm_config.value_type = GM_VALUE_F32) -----------------------------

# heavy_L0 takes tau = 32: with 4-byte values Eq. (6) gives no multisplit chunk
# count at tau = 16 (n_chunksMax < 1), and the planner rejects it as the oracle does
F32_FORCED = [("heavy_L0", {"tau": 32}) if f[0] == "heavy_L0" else f for f in FORCED
              if f[0] in ("auto", "heavy_L0", "heavy_L1", "heavy_L2", "heavy_L3", "unfused", "batched",
                          "L1_wide_chunks", "L1_outer", "L1_rowwise")]


@pytest.mark.parametrize("name,cfg", F32_FORCED, ids=[f[0] for f in F32_FORCED])
@pytest.mark.parametrize("values", ["uniform", "int"])
def test_f32_forced_paths(name, cfg, values):
    """Every pipeline and hierarchy depth with float values."""
    A = gi.rmat(10, 8, seed=1, values=values)
    info = check_full_f32(A, A, exact=values == "int", **cfg)
    if name != "auto":
        assert info.n_heavy_rows > 0


@pytest.mark.parametrize("seed", range(3))
def test_f32_random_irregular(seed):
    """Unsorted rows with repeated columns and explicit zeros (the row-order
    pipeline then splits each tile in shared memory), float values."""
    A = gi.random_csr(64, 90, 0.3, seed, values="int", unsorted=True, duplicates=True, explicit_zeros=True,
                      empty_rows=0.2)
    B = gi.random_csr(90, 70, 0.3, seed + 50, values="int", unsorted=True, duplicates=True, explicit_zeros=True,
                      empty_rows=0.2)
    check_full_f32(A, B, exact=True, tau=2, dense_width=4, n_chunks_max=2)


@pytest.mark.parametrize("scale", [14, 16])
def test_f32_planner_defaults_on_rmat(scale):
    """Default float plan: tau = 14528 and chunks of 32768 columns (Sec. III-D with
    s_C.val = 4); scale 14 needs no multisplit level, scale 16 has two chunks."""
    A = gi.rmat(scale, 16, seed=scale)
    u = oracle.ip_counts(A, A)
    info = check_full_f32(A, A)
    assert info.params.tau == 14528 and info.params.dense_width == 32768
    assert info.n_heavy_rows == int((u > 14528).sum()) > 0
    assert info.params.n_levels == (0 if scale == 14 else 1)


def test_f32_light_rows_laplacian():
    A = gi.laplacian_2d(64)
    check_full_f32(A, A, exact=True)


# --- the workloads ------------------------------------------------------------------

def test_workload_rmat10_fp64_and_int():
    A = gi.named_workload("rmat10")
    check_full(A, A)
    Ai = gi.named_workload("rmat10_int")
    check_full(Ai, Ai, exact=True)


def test_workload_laplacian_1024():
    A = gi.named_workload("laplace1024")
    info = check_full(A, A, exact=True)
    assert info.c_nnz == 13_611_012 and info.n_heavy_rows == 0


def test_workload_erdos_renyi_2_21():
    A = gi.named_workload("er21")
    info = check_full(A, A)
    assert info.ip_total == 64 << 21


def _sampled_check(name, n_random=400, seed=0, f32=False):
    A = gi.named_workload(name)
    if f32:
        A = rounded_to_f32(A)
    u = oracle.ip_counts(A, A)
    Ad = binding.to_device(A, dtype=np.float32 if f32 else None)
    C, info = binding.spgemm(Ad, Ad, return_info=True)
    torch.cuda.synchronize()
    assert info.ip_total == int(u.sum()) and info.n_heavy_rows == int((u > info.params.tau).sum())
    check_invariants(C, u)
    rng = np.random.default_rng(seed)
    heavy = np.nonzero(u > info.params.tau)[0]
    light = np.nonzero((u > 0) & (u <= info.params.tau))[0]
    top = np.argsort(u)[-6:]
    rows = np.unique(np.concatenate([top, rng.choice(heavy, min(n_random, heavy.size), replace=False),
                                     rng.choice(light, min(n_random, light.size), replace=False)]))
    ref = oracle.spgemm_rows(A, A, rows)
    srp, col, val = gather_rows(C, rows)
    if f32:
        ones = ones_like_csr(A)
        assert_matches_f32(ref, oracle.spgemm_rows(ones, ones, rows), srp, col, val)
    else:
        assert_matches(ref, srp, col, val)
    return info


def _full_streamed_check(A, C, block_rows):
    """Every row of C against the oracle, one block of rows at a time, so that
    neither the oracle's C nor the GPU's is ever whole on the host."""
    rp = C.row_ptr.cpu().numpy()
    assert rp[0] == 0 and rp[-1] == C.col.numel()
    for r0 in range(0, A.n_rows, block_rows):
        r1 = min(A.n_rows, r0 + block_rows)
        ref = oracle.spgemm_rows(A, A, np.arange(r0, r1))
        lo, hi = int(rp[r0]), int(rp[r1])
        assert_matches(ref, rp[r0:r1 + 1] - lo, C.col[lo:hi].cpu().numpy(), C.val[lo:hi].cpu().numpy())


@pytest.mark.slow
def test_workload_rmat18_every_row():
    """R-MAT scale 18, edge factor 16 (2.9e9 products, 1.28e9 entries of C): every
    row of C compared with the oracle, structure bit-exact, values within
    1e-12 * sum|ab|."""
    A = gi.named_workload("rmat18")
    Ad = binding.to_device(A)
    C, info = binding.spgemm(Ad, Ad, return_info=True)
    torch.cuda.synchronize()
    assert info.n_heavy_rows > 0 and info.params.n_levels == 1
    _full_streamed_check(A, C, 8192)


def _stratified_rows(u, tau, n_heavy, n_light, rng):
    """Rows drawn evenly from ten strata of u among the heavy rows and among the
    light rows (so every chunk-size class and both heavy batches appear), plus the
    six rows with the most products."""
    picks = [np.argsort(u)[-6:]]
    for sel, n in ((u > tau, n_heavy), ((u > 0) & (u <= tau), n_light)):
        ids = np.nonzero(sel)[0]
        order = ids[np.argsort(u[ids], kind="stable")]
        for part in np.array_split(order, 10):
            if part.size:
                picks.append(rng.choice(part, min(part.size, n // 10), replace=False))
    return np.unique(np.concatenate(picks))


@pytest.mark.slow
def test_workload_rmat20_50k_rows():
    """R-MAT scale 20, edge factor 16 (the benchmark workload): 25,000 heavy and
    25,000 light rows, stratified by their products, compared row by row with the
    oracle over each row's full extent; every row checked for the properties that
    hold at any size (sorted, in range, at most u(i) entries). The opt-in
    GM_FULL_PARITY_20=1 runs test_workload_rmat20_every_row instead of sampling."""
    A = gi.named_workload("rmat20")
    u = oracle.ip_counts(A, A)
    Ad = binding.to_device(A)
    C, info = binding.spgemm(Ad, Ad, return_info=True)
    torch.cuda.synchronize()
    assert info.ip_total == int(u.sum()) and info.n_heavy_rows == int((u > info.params.tau).sum())
    assert info.n_batches >= 2
    check_invariants(C, u)
    rows = _stratified_rows(u, info.params.tau, 25000, 25000, np.random.default_rng(20))
    assert rows.size >= 50000
    for grp in np.array_split(rows, max(1, rows.size // 2000)):
        ref = oracle.spgemm_rows(A, A, grp)
        srp, col, val = gather_rows(C, grp)
        assert_matches(ref, srp, col, val)


@pytest.mark.slow
@pytest.mark.skipif(os.environ.get("GM_FULL_PARITY_20") != "1", reason="opt-in: about 6 minutes of oracle time")
def test_workload_rmat20_every_row():
    """Every row of the scale-20 product (9.7e9 entries of C) against the oracle,
    streamed in blocks of rows."""
    A = gi.named_workload("rmat20")
    Ad = binding.to_device(A)
    C = binding.spgemm(Ad, Ad)
    torch.cuda.synchronize()
    _full_streamed_check(A, C, 16384)


@pytest.mark.slow
def test_workload_rmat20_f32_sampled():
    """The benchmark workload with float values, as `bench.py --dtype f32` runs it:
    tau 14528, 32 level-0 chunks, sampled rows against the oracle."""
    info = _sampled_check("rmat20", n_random=150, f32=True)
    assert info.params.tau == 14528 and list(info.params.v_chunks[:1]) == [32] and info.n_heavy_rows > 0


# --- index types (gm_config.index_type) ---------------------------------------------

# (name, row-pointer dtype, column dtype) at the interface
INDEX_TYPES = [("rowptr32", np.int32, np.int32), ("col64", np.int64, np.int64), ("both", np.int32, np.int64)]
INDEX_PLANS = ["auto", "heavy_L0", "heavy_L2", "L2_outer", "L1_rowwise_256"]


def _index_flags(rp_dt, col_dt):
    return (binding.GM_INDEX_ROWPTR32 if rp_dt == np.int32 else 0) | (binding.GM_INDEX_COL64 if col_dt == np.int64
                                                                    else 0)


def _run_indexed(A, B, rp_dt, col_dt, dtype=None, **cfg):
    Ad = binding.to_device(A, dtype=dtype, row_ptr_dtype=rp_dt, col_dtype=col_dt)
    Bd = Ad if B is A else binding.to_device(B, dtype=dtype, row_ptr_dtype=rp_dt, col_dtype=col_dt)
    C, info = binding.spgemm(Ad, Bd, binding.make_config(**cfg) if cfg else None, return_info=True)
    torch.cuda.synchronize()
    rp, col, val = C.row_ptr.cpu().numpy(), C.col.cpu().numpy(), C.val.cpu().numpy()
    assert rp.dtype == rp_dt and col.dtype == col_dt
    assert info.index_type == _index_flags(rp_dt, col_dt)
    return rp, col, val, info


@pytest.mark.parametrize("name,rp_dt,col_dt", INDEX_TYPES, ids=[t[0] for t in INDEX_TYPES])
@pytest.mark.parametrize("plan", INDEX_PLANS)
def test_index_types_forced_paths(name, rp_dt, col_dt, plan):
    """int32 row pointers and int64 columns at the interface, A*A (A and B share
    their converted copies): structure and integer values equal to the oracle's
    through every hierarchy depth and pipeline."""
    cfg = dict(FORCED)[plan]
    A = gi.rmat(10, 8, seed=1, values="int")
    rp, col, val, info = _run_indexed(A, A, rp_dt, col_dt, **cfg)
    if plan != "auto":
        assert info.n_heavy_rows > 0
    assert_matches(oracle.spgemm(A, A), rp, col, val, exact=True)


@pytest.mark.parametrize("name,rp_dt,col_dt", INDEX_TYPES, ids=[t[0] for t in INDEX_TYPES])
def test_index_types_distinct_operands(name, rp_dt, col_dt):
    """A*B with separate arrays (each converted on its own), unsorted rows with
    repeated columns and explicit zeros, fp64 and float values."""
    A = gi.random_csr(64, 90, 0.3, 7, values="int", unsorted=True, duplicates=True, explicit_zeros=True,
                      empty_rows=0.2)
    B = gi.random_csr(90, 70, 0.3, 8, values="int", unsorted=True, duplicates=True, explicit_zeros=True,
                      empty_rows=0.2)
    ref = oracle.spgemm(A, B)
    for dtype in (None, np.float32):
        rp, col, val, _ = _run_indexed(A, B, rp_dt, col_dt, dtype=dtype, tau=2, dense_width=4, n_chunks_max=2)
        assert_matches(ref, rp, col, val.astype(np.float64), exact=True)
    A, B = gi.named_pair("rmatAB_s13_a4_b8", seed=2)
    rp, col, val, info = _run_indexed(A, B, rp_dt, col_dt)
    assert info.n_heavy_rows > 0
    assert_matches(oracle.spgemm(A, B), rp, col, val)


def test_col64_columns_out_of_range_are_reported():
    """int64 columns outside [0, n_cols) -- also ones whose low 32 bits would be in
    range -- are reported as GM_ERR_BAD_INDEX, in A and in B."""
    A = gi.random_csr(10, 10, 0.4, 1)
    good = binding.to_device(A, col_dtype=np.int64)
    for v in (10, -1, (1 << 31) + 3, (1 << 32) + 2):
        col = A.col.astype(np.int64)
        col[3] = v
        bad = binding.DeviceCSR(A.n_rows, A.n_cols, good.row_ptr, torch.from_numpy(col).cuda(), good.val)
        for lhs, rhs in ((bad, good), (good, bad)):
            with pytest.raises(binding.GmError) as e:
                binding.spgemm(lhs, rhs)
            assert e.value.status == 9


@pytest.mark.slow
def test_rowptr32_overflow_is_reported():
    """C = A*A of the scale-20 R-MAT has 9,708,253,274 entries: int32 row pointers
    cannot hold C.rowPtr, so symbolic returns GM_ERR_INDEX_OVERFLOW with C.nnz on
    the host, writes nothing, and takes no further call."""
    import ctypes
    A = gi.named_workload("rmat20")
    Ad = binding.to_device(A, row_ptr_dtype=np.int32)
    plan = binding.gm_spgemm_analyze(Ad, Ad)
    try:
        c_rp = torch.full((A.n_rows + 1,), -7, dtype=torch.int32, device="cuda")
        nnz = ctypes.c_int64(-1)
        lib = binding.load()
        assert lib.gm_spgemm_symbolic(plan, c_rp.data_ptr(), ctypes.byref(nnz)) == 3
        assert nnz.value == 9_708_253_274
        assert bool((c_rp == -7).all())
        assert lib.gm_spgemm_symbolic(plan, c_rp.data_ptr(), ctypes.byref(nnz)) == 8
    finally:
        binding.gm_spgemm_plan_destroy(plan)


def test_c_program_through_the_abi(tmp_path):
    """C = A*B computed by a plain C program (tests/c_abi_driver.c: CUDA runtime
    copies, analyze / symbolic / numeric with a NULL config, no Python on the
    path) matches the oracle: A*A with heavy and light rows, and a distinct A*B."""
    import subprocess
    from tests.c_driver import build_c_driver, read_csr, write_csr
    exe = build_c_driver(str(tmp_path))
    A = gi.rmat(12, 16, seed=4)
    A2, B2 = gi.named_pair("rmatAB_s13_a4_b8", seed=2)
    for a, b in ((A, A), (A2, B2)):
        fa, fb, fc = (str(tmp_path / n) for n in ("a.bin", "b.bin", "c.bin"))
        write_csr(fa, a)
        write_csr(fb, b)
        out = subprocess.run([exe, fa, fb, fc], capture_output=True, text=True, timeout=120)
        assert out.returncode == 0, out.stderr
        C = read_csr(fc)
        assert C.row_ptr[0] == 0
        assert_matches(oracle.spgemm(a, b), C.row_ptr, C.col, C.val)
    assert " heavy 0 " not in out.stdout
    # the row split of the multi-GPU run, its parts one after another from C
    for parts in (2, 5):
        write_csr(fa, A)
        write_csr(fb, A)
        out = subprocess.run([exe, fa, fb, fc, str(parts)], capture_output=True, text=True, timeout=120)
        assert out.returncode == 0, out.stderr
        assert f"parts {parts}" in out.stdout and " heavy 0 " not in out.stdout
        C = read_csr(fc)
        assert_matches(oracle.spgemm(A, A), C.row_ptr, C.col, C.val)


@pytest.mark.parametrize("values", ["uniform", "int"])
def test_light_chunks_wider_than_65536_columns(values):
    """C.m = 2^19 with chunks of 4 per level down to 4096 columns: four levels
    (131072, 32768, 8192, 4096 columns). The heavy rows' level-0 chunks hold about
    750 elements, below tau, so they leave the hierarchy as light chunks 131072
    columns wide; the bitmap-rank block accumulator then keeps each rank's column
    in 32 bits (16 bits hold chunk-local columns only up to 65536)."""
    rng = np.random.default_rng(17)
    n_mid, n_cols = 3000, 1 << 19

    def rand_csr(n_rows, n_c, per_row):
        rp = np.arange(n_rows + 1, dtype=np.int64) * per_row
        col = np.concatenate([np.sort(rng.choice(n_c, per_row, replace=False)) for _ in range(n_rows)])
        val = (rng.integers(-3, 4, col.size) if values == "int" else rng.uniform(-1, 1, col.size)).astype(np.float64)
        return gi.CSR(n_rows, n_c, rp, col.astype(np.int32), val)

    A = rand_csr(300, n_mid, 30)
    B = rand_csr(n_mid, n_cols, 100)
    info = check_full(A, B, exact=values == "int", tau=2048, dense_width=4096, n_chunks_max=4)
    assert info.params.n_levels == 4 and info.params.widths[0] == 131072 and info.n_heavy_rows > 250


@pytest.mark.parametrize("values", ["uniform", "int", "f32"])
def test_light_rows_over_several_column_windows(values):
    """C.m = 2^21 + 4099: a light row's whole bitmap (256 KB) does not fit beside
    its values, so the numeric light kernel takes the columns in windows of 2^20
    columns, the last one ragged. Every row has about 4000 products (light), so
    each window lists, counts, ranks, writes and clears only its touched groups."""
    rng = np.random.default_rng(23)
    n_mid, n_cols = 5000, (1 << 21) + 4099

    def rand_csr(n_rows, n_c, lo, hi):
        per = rng.integers(lo, hi + 1, n_rows)
        rp = np.concatenate([[0], np.cumsum(per)]).astype(np.int64)
        col = np.concatenate([np.sort(rng.choice(n_c, k, replace=False)) for k in per])
        val = (rng.integers(-3, 4, col.size) if values == "int" else rng.uniform(-1, 1, col.size)).astype(np.float64)
        return gi.CSR(n_rows, n_c, rp, col.astype(np.int32), val)

    A = rand_csr(400, n_mid, 10, 60)  # u <= 60 * 140 < tau
    B = rand_csr(n_mid, n_cols, 60, 140)
    B.col[B.row_ptr[7]] = n_cols - 1  # the last column, in the ragged window
    B.col[B.row_ptr[7]:B.row_ptr[8]].sort()
    if values == "f32":
        info = check_full_f32(A, B)
    else:
        info = check_full(A, B, exact=values == "int")
    assert info.n_heavy_rows == 0 and info.n_light_rows == 400


OVERLAP_CASES = [f for f in FORCED if f[0] in ("auto", "heavy_L1", "heavy_L2", "L1_outer", "L1_rowwise_batched")]


@pytest.mark.parametrize("name,cfg", OVERLAP_CASES, ids=[f[0] for f in OVERLAP_CASES])
@pytest.mark.parametrize("values", ["uniform", "int"])
def test_light_and_heavy_rows_on_two_streams(name, cfg, values):
    """GM_FLAG_OVERLAP: the light rows run on the plan's second stream while the
    heavy rows run on its own; the result is the oracle's."""
    A = gi.rmat(12, 8, seed=6, values=values)
    info = check_full(A, A, exact=values == "int", flags=binding.GM_FLAG_OVERLAP, **cfg)
    assert info.n_light_rows > 0 and (name == "auto" or info.n_heavy_rows > 0)


def test_two_streams_on_every_light_bin():
    A, B = _light_rows_case(1 << 20, 5)
    check_full(A, B, exact=True, flags=binding.GM_FLAG_OVERLAP)
