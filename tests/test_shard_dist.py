"""The row split of one product over several ranks, on CPU with gloo ranks and
the oracle as each rank's compute: the ranks split A's rows with the oracle's
row_split, each computes its rows of C, they all-gather their C.nnz through the
package's host logic (shard.rank_offsets, the one exchange of the split) and
shift their row pointers; the pieces put together equal the oracle's whole C."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, scale, out):
    os.environ.update({"CUDA_VISIBLE_DEVICES": ""})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from sparse_gemm_irregular_gm_gb300 import inputs as gi, shard
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        A = gi.rmat(scale, 8, seed=11, values="int")
        bounds = oracle.row_split(oracle.ip_counts(A, A), world)
        r0, r1 = int(bounds[rank]), int(bounds[rank + 1])
        part = oracle.spgemm_rows(A, A, np.arange(r0, r1))
        base, nnz_all = shard.rank_offsets(part.nnz)
        rp = part.row_ptr + base  # the rank's row pointers inside the whole C
        pieces = [None] * world
        dist.all_gather_object(pieces, (r0, r1, rp, part.col, part.val, base, nnz_all))
        if rank == 0:
            out["pieces"] = pieces
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_row_shards_put_together_equal_the_whole_product(world):
    sys.path.insert(0, ROOT)
    import oracle
    from sparse_gemm_irregular_gm_gb300 import inputs as gi
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    scale = 9
    mp.start_processes(_rank_main, args=(world, _free_port(), scale, out), nprocs=world, join=True,
                       start_method="spawn")
    pieces = out["pieces"]
    A = gi.rmat(scale, 8, seed=11, values="int")
    ref = oracle.spgemm(A, A)
    nnz_all = pieces[0][6]
    assert nnz_all == [p[4].size for p in pieces]
    rows = 0
    for q, (r0, r1, rp, col, val, base, every) in enumerate(pieces):
        assert every == nnz_all and base == sum(nnz_all[:q]) and r0 == rows
        rows = r1
        np.testing.assert_array_equal(rp, ref.row_ptr[r0:r1 + 1])  # shifted pointers are the whole C's
        np.testing.assert_array_equal(col, ref.col[rp[0]:rp[-1]])
        np.testing.assert_array_equal(val, ref.val[rp[0]:rp[-1]])  # integer values: exact
    assert rows == A.n_rows and sum(nnz_all) == ref.nnz


def test_single_rank_offsets_need_no_process_group():
    sys.path.insert(0, ROOT)
    from sparse_gemm_irregular_gm_gb300 import shard
    assert shard.rank_offsets(12345) == (0, [12345])
