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
