"""C = A * B spread over several GPUs by rows of A (one process per GPU).

Every rank holds A and B whole in its own GPU's memory and computes one range of
C's rows through the library: ``gm_spgemm_row_split`` cuts A's rows into ranges
of about equal intermediate products, ``gm_spgemm_analyze_rows`` and the usual
symbolic and numeric calls compute the rank's rows, and ``gm_row_ptr_shift``
moves the rank's row pointers behind the entries of the ranks before it. The
only exchange between ranks is one all-gather of each rank's C.nnz (8 bytes a
rank). C stays distributed: rank q owns rows [bounds[q], bounds[q+1]) and the
entries [base_q, base_q + nnz_q) of the whole product, and its row pointers are
those of the whole C.

Everything here is host-side orchestration; every step on the data runs in the
library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

from . import binding


@dataclass
class RowShard:
    """One rank's part of C = A * B."""

    row_begin: int
    row_end: int
    base: int                 # entries of C in the rows before row_begin
    nnz_all: list             # C.nnz of every rank's rows, rank order
    C: binding.DeviceCSR      # rows [row_begin, row_end); row pointers of the whole C
    info: object = None       # gm_plan_info of the rank's plan (with return_info)


def _rank_world(group=None):
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            return dist.get_rank(group), dist.get_world_size(group)
    except ImportError:
        pass
    return 0, 1


def rank_offsets(local_nnz: int, group=None):
    """All-gather of every rank's C.nnz (one int64 a rank). Returns (base, nnz_all):
    the entries of C before this rank's rows, and the list of every rank's count."""
    rank, world = _rank_world(group)
    if world == 1:
        return 0, [int(local_nnz)]
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" \
        else torch.device("cpu")
    mine = torch.tensor([int(local_nnz)], dtype=torch.int64, device=dev)
    every = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(every, mine, group=group)
    nnz_all = [int(t.item()) for t in every]
    return sum(nnz_all[:rank]), nnz_all


def row_bounds(A: binding.DeviceCSR, B: binding.DeviceCSR, n_parts: int, cfg=None, stream=None):
    """The library's split of A's rows into n_parts ranges of about equal products."""
    return binding.gm_spgemm_row_split(A, B, n_parts, cfg, stream)


def spgemm_row_shard(A: binding.DeviceCSR, B: binding.DeviceCSR, cfg=None, group=None, stream=None,
                     bounds=None, return_info: bool = False) -> RowShard:
    """This rank's rows of C = A * B (see the module docstring). ``bounds`` may be
    given (the same on every rank); otherwise the library computes them."""
    rank, world = _rank_world(group)
    if bounds is None:
        bounds = row_bounds(A, B, world, cfg, stream) if world > 1 else [0, A.n_rows]
    r0, r1 = int(bounds[rank]), int(bounds[rank + 1])
    C, info = binding.spgemm(A, B, cfg, stream, rows=(r0, r1), return_info=True)
    base, nnz_all = rank_offsets(C.nnz, group)
    if base:
        binding.gm_row_ptr_shift(C.row_ptr, base, stream)
    return RowShard(r0, r1, base, nnz_all, C, info if return_info else None)
