"""Workspace allocation failure, injected on the host through the allocator hooks
(gm_set_allocator): the k-th allocation of a product returns NULL, for every k
from the first to the last. Each product must then either succeed (an arena
that cannot be had makes the plan halve its batch budget and plan again) and
equal the oracle's C, or stop with GM_ERR_OOM; either way every workspace block
is handed back by the time the plan is destroyed. Nothing here makes the GPU
fault: the library checks each allocation before a kernel can see the buffer.
"""
import ctypes

import numpy as np
import pytest

import oracle
from sparse_gemm_irregular_gm_gb300 import binding, inputs as gi
from tests.gpu_common import assert_matches

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GM_ERR_OOM = 4


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    lib = binding.load()
    yield lib
    binding.use_torch_allocator(True)


class Hooks:
    """Workspace from torch's caching allocator, failing the fail_at-th request."""

    def __init__(self, fail_at=0):
        self.calls = 0
        self.fail_at = fail_at
        self.live = {}

    def alloc(self, ctx, nbytes, stream):
        self.calls += 1
        if self.calls == self.fail_at:
            return None
        p = torch.cuda.caching_allocator_alloc(int(nbytes), torch.cuda.current_device(), stream or 0)
        self.live[p] = int(nbytes)
        return p

    def free(self, ctx, ptr, nbytes, stream):
        assert self.live.pop(ptr) == int(nbytes), "a block came back with another size"
        torch.cuda.caching_allocator_delete(ptr)

    def install(self, lib):
        self.cbs = (binding._ALLOC_T(self.alloc), binding._FREE_T(self.free), binding._AVAIL_T(lambda ctx: -1))
        lib.gm_set_allocator(*[ctypes.cast(f, ctypes.c_void_p) for f in self.cbs], None)


CASES = [
    ("one_level_batched", {"tau": 64, "dense_width": 256, "n_chunks_max": 16, "workspace_cap_bytes": 12 << 20}),
    ("two_levels_outer", {"tau": 64, "dense_width": 64, "n_chunks_max": 4, "workspace_cap_bytes": 16 << 20,
                          "pipeline": binding.GM_PIPE_FUSED_HISTO}),
    ("two_streams", {"tau": 64, "dense_width": 256, "n_chunks_max": 16, "flags": binding.GM_FLAG_OVERLAP}),
]


@pytest.mark.parametrize("name,cfg", CASES, ids=[c[0] for c in CASES])
def test_every_allocation_failing_once(lib, name, cfg):
    A = gi.rmat(11, 8, seed=8, values="int")
    ref = oracle.spgemm(A, A)
    Ad = binding.to_device(A)
    config = binding.make_config(**cfg)
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    counting = Hooks()
    counting.install(lib)
    C = binding.spgemm(Ad, Ad, config)
    torch.cuda.synchronize()
    n_allocs = counting.calls
    assert n_allocs > 10 and not counting.live
    del C
    outcomes = {"ok": 0, "oom": 0}
    for k in range(1, n_allocs + 1):
        hooks = Hooks(fail_at=k)
        hooks.install(lib)
        try:
            C = binding.spgemm(Ad, Ad, config)
            torch.cuda.synchronize()
            assert_matches(ref, C.row_ptr.cpu().numpy(), C.col.cpu().numpy(), C.val.cpu().numpy(), exact=True)
            del C
            outcomes["ok"] += 1
        except binding.GmError as e:
            assert e.status == GM_ERR_OOM, f"allocation {k} of {n_allocs}: {e}"
            outcomes["oom"] += 1
        torch.cuda.synchronize()
        assert not hooks.live, f"allocation {k} failing left {len(hooks.live)} workspace blocks behind"
        assert torch.cuda.memory_allocated() == base, f"allocation {k} failing left device memory behind"
    assert outcomes["oom"] > 0
    binding.use_torch_allocator(True)
