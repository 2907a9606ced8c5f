"""bench.py's multi-rank plumbing on CPU: two gloo ranks set up the process
group from the launcher's environment, meet at the barrier, and agree on the
slowest rank's time (the timing rule for N > 1: max over ranks)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "CUDA_VISIBLE_DEVICES": ""})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(None)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(times[rank], w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    times = [0.25, 0.75]
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 0.75, 1: 0.75}


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    bench.barrier(1)


def test_captured_traffic_only_while_sources_match(tmp_path, monkeypatch):
    """bench.py reports the committed DRAM-byte capture only for its workload and
    stage, and only while the kernel sources hash as they did at capture time."""
    import hashlib
    import json
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    rec = {"workload": "rmat20", "stages": {"num_heavy": {"dram_read_bytes": 7, "dram_write_bytes": 5}},
           "sources_sha256": {str(src): hashlib.sha256(b"kernel v1").hexdigest()}}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.captured_traffic("rmat20", "num_heavy") == 12
    assert bench.captured_traffic("rmat18", "num_heavy") is None
    assert bench.captured_traffic("rmat20", "multisplit") is None
    src.write_text("kernel v2")
    assert bench.captured_traffic("rmat20", "num_heavy") is None


def test_byte_model_counts_a_and_c_at_the_interface_widths():
    """With int32 row pointers and int64 columns the byte model counts A and C
    (read once, written once) at those widths; the per-stage bytes, which are
    the path's own element layouts, do not change."""
    from types import SimpleNamespace
    sys.path.insert(0, ROOT)
    import bench
    A = SimpleNamespace(n_rows=1000, nnz=16000)
    info = SimpleNamespace(ip_heavy=10 ** 6, params=SimpleNamespace(n_levels=1))
    nnz_c = 50000
    base, st0 = bench.byte_model(info, A, nnz_c, True, 8, 2)
    both, st1 = bench.byte_model(info, A, nnz_c, True, 8, 2, 4, 8)
    # A twice (read by the count and the expansion) and C once: -4 B a row pointer, +4 B a column
    assert both - base == 2 * (-4 * 1001 + 4 * 16000) + (-4 * 1001 + 4 * nnz_c)
    assert st0 == st1
    args = SimpleNamespace(index_type="both")
    assert [d.itemsize for d in bench.index_dtypes(args)] == [4, 8]
    assert set(bench.INDEX_TYPES) == {"default", "rowptr32", "col64", "both"}
