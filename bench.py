#!/usr/bin/env python
"""Benchmark of the gMAGNUS SpGEMM C = A*A on GB300.

Workload: A = R-MAT scale 20 (1,048,576 x 1,048,576), edge factor 16, quadrant
probabilities 0.57/0.19/0.19/0.05, duplicates collapsed, fp64 U[-1,1), seed 1;
C = A*A (2.09e10 intermediate products, 9.7e9 nonzeros). A step is one full
SpGEMM through the C ABI: analyze, symbolic, allocation of C, numeric.

Printed: one JSON line with GFLOP/s = 2 * intermediate products / time, the
roofline of the dominant stage, the whole-path roofline on the method's byte
model, an end-to-end figure with host buffers (inputs copied in, C copied out),
clocks sampled during the timed region and the CPU oracle as a baseline.
``--impl reference`` times the CPU oracle instead (bounded row samples).
Multi-GPU (torchrun): the product is split by rows of A into parts of about
equal intermediate products, one part a GPU (each rank holds A and B whole and
computes its rows of C through the library; the ranks all-gather their C.nnz,
8 bytes each, to place their row pointers); value = the whole product's
2 * products / max time over ranks (strong scaling: the work is fixed).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SpGEMM GFLOP/s (2×intermediate products/s) and % of HBM roofline, 1×GB300"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="rmat20")
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--pipeline", type=int, default=0)
    ap.add_argument("--dtype", choices=["f64", "f32"], default="f64", help="value type of A, B and C")
    ap.add_argument("--index-type", choices=list(INDEX_TYPES), default="default",
                    help="row-pointer / column types of A, B and C at the interface")
    ap.add_argument("--tau", type=int, default=0, help="plan override: heavy-row threshold")
    ap.add_argument("--n-chunks-max", type=int, default=0, help="plan override: chunks per multisplit level")
    ap.add_argument("--dense-width", type=int, default=0, help="plan override: dense accumulator width")
    ap.add_argument("--grid", action="store_true",
                    help="C = A*B over the R-MAT grid of distinct pairs (one JSON line per point)")
    ap.add_argument("--grid-max-scale", type=int, default=0, help="leave out grid points above this scale")
    ap.add_argument("--overlap", action="store_true", help="light rows on a second stream (GM_FLAG_OVERLAP)")
    ap.add_argument("--e2e-parts", type=int, default=4,
                    help="row parts of the end-to-end leg: C of one part is copied out while the next is computed")
    return ap.parse_args()


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_rmat20_ef16_AxA.json")


def captured_traffic(workload: str, stage: str):
    """DRAM bytes (read + write) of one step of `stage`, from the committed ncu
    capture, while the kernel sources still hash as they did then; else None."""
    import hashlib
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        if d["workload"] != workload or stage not in d["stages"]:
            return None
        for rel, digest in d["sources_sha256"].items():
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        st = d["stages"][stage]
        return int(st["dram_read_bytes"]) + int(st["dram_write_bytes"])
    except (OSError, KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, power, reasons = [], [], [], set()
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(self.NAMES, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        os.unlink(self.file.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def byte_model(info, A, nnz_c, rowwise, vb=8, cb=4, rp_b=8, col_b=4):
    """Algorithmic bytes per step.

    Whole path, outer-product pipelines (the method's byte model, one multisplit
    level): read A and B once, C-hat written once (12 B/product), per level a
    histogram read of columns (4) and a multisplit read + write (12 + 12), a
    symbolic column read (4), a numeric read (12), C written once.
    Row-order pipeline: C-hat is never written; the expansion writes each heavy
    product once, already in its level-0 chunk (12), the symbolic pass reads the
    B columns it walks (4) and the numeric pass reads the chunks once (12).
    Per stage: the bytes that stage must move in this implementation (symbolic
    passes carry columns only, numeric passes columns and values; the level-0
    histogram is counted inside the outer product). Element sizes are for vb-byte
    values (12 B for a column and a double, 8 B with floats); the row-order
    pipeline stores chunk-local columns in cb bytes (2: uint16). A and C are
    counted at the interface's widths: rp_b bytes a row pointer, col_b a column.
    """
    e = 4 + vb
    ec = cb + vb
    ip_h = info.ip_heavy
    L = max(1, info.params.n_levels)
    a_bytes = rp_b * (A.n_rows + 1) + (col_b + vb) * A.nnz
    c_bytes = rp_b * (A.n_rows + 1) + (col_b + vb) * nnz_c
    if rowwise:
        b_alg = 2 * a_bytes + ip_h * (ec + 4 + ec) + c_bytes
        stages = {
            "multisplit": ip_h * ec,    # products written once, into their level-0 chunks
            "sym_heavy": ip_h * 4,      # B columns walked
            "num_heavy": ip_h * ec,     # chunk columns and values read (+ C writes, added by the caller)
        }
        return b_alg, stages
    b_alg = 2 * a_bytes + ip_h * (e + L * (4 + e + e) + 4 + e) + c_bytes
    stages = {
        "outer_sym": ip_h * 4,          # C-hat columns written (symbolic pass)
        "outer": ip_h * e,              # C-hat columns and values written (numeric pass)
        "multisplit_sym": ip_h * 8,     # columns read and written
        "multisplit": ip_h * 2 * e,     # columns and values read and written
        "sym_heavy": ip_h * 4,          # chunk columns read
        "num_heavy": ip_h * e,          # chunk columns and values read (+ C writes, added by the caller)
    }
    return b_alg, stages


def log(msg):
    print(f"[bench] {msg}", file=sys.stderr, flush=True)


# In the row-order pipeline three of the library's stage slots time other work
# than their names say: the gather of the heavy rows' A entries (TRANSPOSE), the
# chunk offsets (HISTOGRAM) and the expansion into level-0 chunks (MULTISPLIT).
ROWWISE_STAGE_NAMES = {"transpose": "gather_entries", "histogram": "chunk_offsets", "multisplit": "expansion"}


def stage_label(name: str, rowwise: bool) -> str:
    return ROWWISE_STAGE_NAMES.get(name, name) if rowwise else name


def _read_int(path):
    try:
        with open(path) as f:
            return int(f.read().split()[0])
    except (OSError, ValueError, IndexError):
        return None


def host_available_bytes():
    """Host memory this process may still take: the smaller of the machine's
    MemAvailable and the room left under its cgroup's memory limit."""
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    for limit_f, usage_f in (("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory.current"),
                             ("/sys/fs/cgroup/memory/memory.limit_in_bytes",
                              "/sys/fs/cgroup/memory/memory.usage_in_bytes")):
        limit, usage = _read_int(limit_f), _read_int(usage_f)  # "max" (no limit) reads as None
        if limit is not None and usage is not None and limit < (1 << 60):
            room = max(0, limit - usage)
            avail = room if avail is None else min(avail, room)
            break
    return avail


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _cpu_baseline_child(workload, seed, target_s):
    import oracle
    from sparse_gemm_irregular_gm_gb300 import inputs
    A, B = inputs.named_pair(workload, seed=seed)
    return _cpu_baseline(A, B, oracle.ip_counts(A, B), target_s, seed)


def cpu_baseline(workload, seed, target_s):
    """The oracle timed in a spawned process (its memory is returned when it exits)."""
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(1) as pool:
        return pool.apply(_cpu_baseline_child, (workload, seed, target_s))


def _cpu_baseline(A, B, u, target_s, seed):
    """The oracle, as it stands, on a bounded random sample of A's rows."""
    import numpy as np

    import oracle
    rng = np.random.default_rng(seed)
    order = rng.permutation(A.n_rows)
    csum = np.cumsum(u[order])
    # calibrate on ~2e7 products, then size the sample for target_s seconds
    k = min(A.n_rows, int(np.searchsorted(csum, 2e7)) + 1)
    t0 = time.perf_counter()
    oracle.spgemm_rows(A, B, np.sort(order[:k]))
    rate = float(csum[k - 1]) / max(time.perf_counter() - t0, 1e-3)
    k = int(np.searchsorted(csum, rate * target_s)) + 1
    k = min(k, A.n_rows)
    rows = np.sort(order[:k])
    ip = int(csum[k - 1])
    t0 = time.perf_counter()
    oracle.spgemm_rows(A, B, rows)
    dt = time.perf_counter() - t0
    return {"value": 2.0 * ip / dt / 1e9, "unit": "GFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{k} random rows of the workload ({ip:.3e} of {int(u.sum()):.3e} intermediate products), "
                      f"{dt:.1f} s on the host cores"}


# --index-type: (row-pointer dtype, column dtype) of the arrays handed to the library
INDEX_TYPES = {"default": ("int64", "int32"), "rowptr32": ("int32", "int32"), "col64": ("int64", "int64"),
               "both": ("int32", "int64")}


def index_dtypes(args):
    import numpy as np
    rp, col = INDEX_TYPES[args.index_type]
    return np.dtype(rp), np.dtype(col)


def plan_overrides(args) -> dict:
    """gm_config fields set on the command line (zero keeps the automatic value)."""
    return {k: v for k, v in (("n_chunks_max", args.n_chunks_max), ("dense_width", args.dense_width),
                              ("tau", args.tau)) if v}


def workload_name(args) -> str:
    vals = "fp32 U[-1,1)" if args.dtype == "f32" else "fp64 U[-1,1)"
    idx = "" if args.index_type == "default" else ", %s row pointers, %s columns" % INDEX_TYPES[args.index_type]
    if args.workload == "rmat20":
        return f"A*A, A = R-MAT scale 20, edge factor 16, a=.57 b=.19 c=.19, {vals}, seed 1{idx}"
    if args.dtype == "f64" and not idx:
        return args.workload
    return f"{args.workload} ({vals}{idx})"


def make_step(A, Ad, Bd, cfg, stream):
    """One full SpGEMM through the C ABI: analyze, symbolic, allocation of C, numeric."""
    import torch

    from sparse_gemm_irregular_gm_gb300 import binding

    def step():
        plan = binding.gm_spgemm_analyze(Ad, Bd, cfg, stream)
        c_rp = torch.empty(A.n_rows + 1, dtype=Ad.row_ptr.dtype, device="cuda")
        nnz = binding.gm_spgemm_symbolic(plan, c_rp)
        c_col = torch.empty(nnz, dtype=Ad.col.dtype, device="cuda")
        c_val = torch.empty(nnz, dtype=Ad.val.dtype, device="cuda")
        binding.gm_spgemm_numeric(plan, c_col, c_val)
        info = binding.gm_spgemm_plan_info(plan)
        binding.gm_spgemm_plan_destroy(plan)
        return info, c_rp
    return step


def make_shard_step(Ad, Bd, cfg, stream):
    """This rank's part of the product split by rows (shard.spgemm_row_shard): the
    library's split, the rank's rows through the C ABI, the all-gather of C.nnz
    and the shift of the rank's row pointers."""
    from sparse_gemm_irregular_gm_gb300 import shard

    def step():
        part = shard.spgemm_row_shard(Ad, Bd, cfg, stream=stream, return_info=True)
        return part.info, part.C.row_ptr, (part.row_begin, part.row_end, part.base, sum(part.nnz_all))
    return step


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__
    from sparse_gemm_irregular_gm_gb300 import binding, inputs
    rank, world, local = dist_setup(args)
    __graft_entry__.build()
    A, B = inputs.named_pair(args.workload, seed=args.seed)
    vdt = np.float32 if args.dtype == "f32" else None
    vb = 4 if args.dtype == "f32" else 8
    rp_dt, col_dt = index_dtypes(args)
    Ad = binding.to_device(A, dtype=vdt, row_ptr_dtype=rp_dt, col_dtype=col_dt)
    Bd = Ad if B is A else binding.to_device(B, dtype=vdt, row_ptr_dtype=rp_dt, col_dtype=col_dt)
    flags = binding.GM_FLAG_TIMING | (binding.GM_FLAG_OVERLAP if args.overlap else 0)
    cfg = binding.make_config(flags=flags, pipeline=args.pipeline, **plan_overrides(args))
    if args.dtype == "f32":
        cfg.value_type = binding.GM_VALUE_F32
    stream = torch.cuda.current_stream()
    if world > 1:
        step = make_shard_step(Ad, Bd, cfg, stream)
    else:
        plain = make_step(A, Ad, Bd, cfg, stream)

        def step():
            info, c_rp = plain()
            return info, c_rp, (0, A.n_rows, 0, None)

    log(f"workload {args.workload}: n={A.n_rows} nnz={A.nnz}, {world} rank(s)")
    for w in range(args.warmup):
        t0 = time.perf_counter()
        info, c_rp, _ = step()
        del c_rp
        log(f"warmup {w}: {time.perf_counter() - t0:.3f} s, stages {[round(x, 1) for x in info.stage_ms]}")
    # per-row products and the heavy rows (for the byte model and the CPU sample)
    plan = binding.gm_spgemm_analyze(Ad, Bd, None, stream)
    u = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_IP_COUNTS)
    heavy = binding.gm_spgemm_debug_copy(plan, binding.GM_DBG_HEAVY_ROWS).astype(np.int64)
    binding.gm_spgemm_plan_destroy(plan)

    clocks = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stage_ms = np.zeros(binding.GM_NUM_STAGES)
    launches = 0
    e0.record(stream)
    for _ in range(args.steps):
        info, c_rp, span = step()
        stage_ms += np.array(info.stage_ms[:])
        launches += info.kernel_launches
        last_rp = c_rp
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    stage_ms /= args.steps
    r0, r1, base, nnz_total = span
    rp = last_rp.cpu().numpy().astype(np.int64) - base  # this rank's rows, from 0
    nnz_c = int(rp[-1])  # this rank's entries of C
    mine = heavy[(heavy >= r0) & (heavy < r1)] - r0
    nnz_heavy = int((rp[mine + 1] - rp[mine]).sum())
    del last_rp, c_rp
    nnz_total = nnz_c if nnz_total is None else int(nnz_total)
    flops = 2.0 * float(u.sum())  # the whole product, whatever the number of ranks
    value = flops / (ms / 1e3) / 1e9
    peak, peak_kind = peaks()
    rowwise = info.pipeline == binding.GM_PIPE_ROWWISE
    # byte models of this rank's part (the whole product on one GPU): A's rows of the part, its C
    A_part = type("Part", (), {"n_rows": r1 - r0, "nnz": int(A.row_ptr[r1] - A.row_ptr[r0])})
    b_alg, stage_bytes = byte_model(info, A_part, nnz_c, rowwise, vb, info.chunk_col_bytes or 4,
                                    rp_dt.itemsize, col_dt.itemsize)
    b_method, _ = byte_model(info, A_part, nnz_c, False, vb, 4, rp_dt.itemsize, col_dt.itemsize)
    b_alg, b_method = sum_over_ranks(b_alg, world), sum_over_ranks(b_method, world)
    stage_bytes["num_heavy"] += (4 + vb) * nnz_heavy + 8 * len(mine)
    names = binding.STAGES
    stage_table = {stage_label(names[i], rowwise): round(float(stage_ms[i]), 3)
                   for i in range(len(names)) if stage_ms[i] > 0}
    dom = max(stage_bytes, key=lambda k: stage_ms[names.index(k)])
    dom_s = stage_ms[names.index(dom)] / 1e3
    achieved = stage_bytes[dom] / dom_s / 1e9 if dom_s > 0 else 0.0
    job_peak = peak * world
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": workload_name(args),
                   "n": A.n_rows, "nnz_A": A.nnz, "intermediate_products": int(u.sum()),
                   "heavy_products": int(u[heavy].sum()), "nnz_C": nnz_total, "heavy_rows": int(heavy.size),
                   "levels": info.params.n_levels, "chunks": list(info.params.v_chunks[:info.params.n_levels]),
                   "batches": info.n_batches, "pipeline": binding.PIPELINES[info.pipeline],
                   "plan_overrides": plan_overrides(args) or None,
                   "index_type": None if args.index_type == "default" else args.index_type,
                   "light_rows_stream": "second stream (GM_FLAG_OVERLAP)" if args.overlap else "plan's stream",
                   "parallelism": f"row split over {world} GPUs (parts of equal products, C.nnz all-gather)"
                   if world > 1 else "single GPU",
                   "l2": "inputs and outputs larger than L2 (C alone is %.0f GB)" % ((4 + vb) * nnz_total / 1e9)},
        "roofline": {"bound": "hbm", "kernel": stage_label(dom, rowwise), "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": captured_traffic(args.workload, dom) if args.pipeline == 0 and world == 1 and
                     not plan_overrides(args) and args.dtype == "f64" and args.index_type == "default" and
                     not args.overlap else None,
                     "traffic_note": "DRAM read + write bytes of the stage's kernels in one step (ncu, "
                                     "profiles/traffic_rmat20_ef16_AxA.json); null once they change",
                     "peak_kind": peak_kind, "alg_bytes_per_step": int(stage_bytes[dom])},
        "path_roofline": {"alg_bytes": int(b_alg), "frac": round((b_alg / (job_peak * 1e9)) / (ms / 1e3), 4),
                          "peak": job_peak, "unit": "GB/s", "peak_kind": peak_kind,
                          "model": "the bytes this pipeline must move (the figure the 50% goal is measured on)"},
        "method_roofline": {"alg_bytes": int(b_method),
                            "frac": round((b_method / (job_peak * 1e9)) / (ms / 1e3), 4),
                            "peak": job_peak, "unit": "GB/s", "peak_kind": peak_kind,
                            "model": "equivalent rate on the method's byte model (C-hat written, histogram, "
                                     "multisplit, symbolic and numeric passes over it: 56 B per heavy product "
                                     "at one level); the row-order pipeline skips those passes, so this is "
                                     "not an achieved bandwidth"},
        "stages_ms": stage_table,
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    log("timed: " + json.dumps({k: result[k] for k in ("value", "ms_per_step", "stages_ms", "roofline")}))
    # The CPU leg runs first, in a spawned process whose memory is returned when
    # it exits; the end-to-end leg pins C's size in host memory and runs last.
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(args.workload, args.seed, args.cpu_seconds)
        log("cpu_baseline: " + json.dumps(result["cpu_baseline"]))
    if not args.no_e2e and rank == 0 and world == 1 and B is A:
        result["e2e"] = run_e2e(args, A, cfg, stream, nnz_c, int(u.sum()))
        log("e2e: " + json.dumps(result["e2e"]))
    if rank == 0:
        print(json.dumps(result), flush=True)


# gMAGNUS, Sec. IV-A, Table III (RMat pairs from PaRMAT, B.nnz/B.n = 8):
# (A.nnz/A.n, scale) -> (C.nnz/C.n, C-hat.nnz/C-hat.n); the pages print N/A for the
# larger scales at A.nnz/A.n >= 8, and those points are not in the grid.
TABLE_III = {
    (4, 15): (477.6, 819.9), (4, 16): (633.5, 1068.2), (4, 17): (835.0, 1382.7),
    (4, 18): (1112.7, 1802.7), (4, 19): (1471.9, 2342.3), (4, 20): (1944.1, 3043.1),
    (8, 15): (782.3, 1548.9), (8, 16): (1048.4, 2021.2), (8, 17): (1397.9, 2628.5),
    (8, 18): (1875.6, 3432.7), (8, 19): (2496.0, 4472.1),
    (16, 15): (1233.3, 2841.0), (16, 16): (1679.4, 3746.7), (16, 17): (2267.3, 4911.0),
    (16, 18): (3075.3, 6427.6),
    (32, 15): (1895.6, 5149.9), (32, 16): (2597.7, 6779.1), (32, 17): (3574.5, 8979.8),
    (32, 18): (4896.9, 11805.3),
}


def run_grid(args):
    """C = A*B over the R-MAT grid of the pages' Table III (distinct A and B, B.nnz/B.n = 8):
    one JSON line per point with the measured rate and the statistics next to the
    table's. The table's matrices come from PaRMAT, ours from the R-MAT generator of
    this package with the same quadrant probabilities, so the statistics agree only
    approximately. L2 is flushed before every timed step."""
    import torch

    import __graft_entry__
    from sparse_gemm_irregular_gm_gb300 import binding, inputs
    rank, world, local = dist_setup(args)
    __graft_entry__.build()
    stream = torch.cuda.current_stream()
    cfg = binding.make_config(flags=binding.GM_FLAG_TIMING, pipeline=args.pipeline)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    points = sorted(TABLE_III, key=lambda k: (k[1], k[0]))
    if args.grid_max_scale:
        points = [p for p in points if p[1] <= args.grid_max_scale]
    for a_density, scale in points:
        name = f"rmatAB_s{scale}_a{a_density}_b8"
        A, B = inputs.named_pair(name, seed=args.seed)
        Ad, Bd = binding.to_device(A), binding.to_device(B)
        step = make_step(A, Ad, Bd, cfg, stream)
        for _ in range(max(1, args.warmup)):
            info, c_rp = step()
            del c_rp
        times = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            info, c_rp = step()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
            nnz_c = int(c_rp[-1].item())
            del c_rp
        ms = max_over_ranks(statistics.median(times), world)
        c_n, chat_n = TABLE_III[(a_density, scale)]
        line = {
            "grid": name, "metric": METRIC, "value": round(world * 2.0 * info.ip_total / ms / 1e6, 3),
            "unit": "GFLOP/s", "ms_per_step": round(ms, 3), "steps": args.steps, "n_gpus": world,
            "dtype": "f64", "data": "synthetic", "l2": "flushed before each timed step",
            "n": A.n_rows, "A_nnz_per_row": round(A.nnz / A.n_rows, 2), "B_nnz_per_row": round(B.nnz / B.n_rows, 2),
            "C_nnz_per_row": round(nnz_c / A.n_rows, 1), "Chat_nnz_per_row": round(info.ip_total / A.n_rows, 1),
            "table_III": {"C_nnz_per_row": c_n, "Chat_nnz_per_row": chat_n},
            "heavy_rows": info.n_heavy_rows, "chunks": list(info.params.v_chunks[:info.params.n_levels]),
            "pipeline": binding.PIPELINES[info.pipeline],
            "stages_ms": {binding.STAGES[i]: round(float(x), 3) for i, x in enumerate(info.stage_ms) if x > 0},
        }
        if rank == 0:
            print(json.dumps(line), flush=True)
        del Ad, Bd, step
        torch.cuda.empty_cache()


def run_e2e(args, A, cfg, stream, nnz_c, ip_total):
    """Same metric with host buffers: copy A in from pinned memory, run, copy C out."""
    import torch

    vb = 4 if args.dtype == "f32" else 8
    rp_dt, col_dt = index_dtypes(args)
    h2d = (A.n_rows + 1) * rp_dt.itemsize + A.nnz * (col_dt.itemsize + vb)
    d2h = (A.n_rows + 1) * rp_dt.itemsize + nnz_c * (col_dt.itemsize + vb)
    avail = host_available_bytes()
    if avail is not None and d2h + h2d > 0.8 * avail:
        return {"value": None, "unit": "GFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "skipped": f"C needs {d2h / 1e9:.0f} GB of pinned host memory, {avail / 1e9:.0f} GB available"}
    try:
        return _run_e2e_pinned(args, A, cfg, stream, nnz_c, ip_total, vb, h2d, d2h)
    except RuntimeError as e:  # pinned allocation refused: report, do not lose the line
        return {"value": None, "unit": "GFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "skipped": f"pinned host buffers: {str(e).splitlines()[0][:200]}"}
    finally:
        # return the pinned pages to the system (torch keeps freed pinned blocks cached)
        import gc
        gc.collect()
        if hasattr(torch._C, "_host_emptyCache"):
            torch._C._host_emptyCache()


def _gpu_numa_cpus():
    """CPUs of the NUMA node the current GPU hangs off (sysfs through the GPU's PCI
    id), or None when the system does not say."""
    import torch
    try:
        bus = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                              "-i", str(torch.cuda.current_device())], capture_output=True, text=True,
                             timeout=30).stdout.strip()
        dom, rest = bus.split(":", 1)
        with open(f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest.lower()}/numa_node") as f:
            node = int(f.read().strip())
        if node < 0:
            return None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            cpus = set()
            for part in f.read().strip().split(","):
                lo, _, hi = part.partition("-")
                cpus.update(range(int(lo), int(hi or lo) + 1))
        return cpus or None
    except (OSError, ValueError, subprocess.SubprocessError):
        return None


def _pinned(n, dtype, cpus):
    """An empty pinned host tensor, its pages first touched from the GPU's NUMA node
    when that is known (the default local policy then places them there)."""
    import torch
    if not cpus:
        return torch.empty(n, dtype=dtype, pin_memory=True)
    old = os.sched_getaffinity(0)
    try:
        os.sched_setaffinity(0, cpus)
        return torch.empty(n, dtype=dtype, pin_memory=True)
    finally:
        os.sched_setaffinity(0, old)


def _run_e2e_pinned(args, A, cfg, stream, nnz_c, ip_total, vb, h2d, d2h):
    """Inputs copied in, then the product in args.e2e_parts row parts (the library's
    row split): while part q+1 is computed, part q of C is copied out on two copy
    streams. One step ends when all of C is in host memory."""
    import numpy as np
    import torch

    from sparse_gemm_irregular_gm_gb300 import binding
    rp_dt, col_dt = index_dtypes(args)
    cpus = _gpu_numa_cpus()
    h_rp = torch.from_numpy(A.row_ptr.astype(rp_dt)).pin_memory()
    h_col = torch.from_numpy(A.col.astype(col_dt)).pin_memory()
    h_val = torch.from_numpy(A.val.astype(np.float32) if vb == 4 else A.val).pin_memory()
    t0 = time.perf_counter()
    o_rp = _pinned(A.n_rows + 1, h_rp.dtype, cpus)
    o_col = _pinned(nnz_c, h_col.dtype, cpus)
    o_val = _pinned(nnz_c, h_val.dtype, cpus)
    log(f"e2e: pinned {d2h / 1e9:.1f} GB of host memory in {time.perf_counter() - t0:.1f} s "
        f"({'on the GPU NUMA node' if cpus else 'NUMA node of the GPU unknown'})")

    torch.cuda.empty_cache()  # let this leg's own allocation sizes form the cache
    d_rp = torch.empty_like(h_rp, device="cuda")
    d_col = torch.empty_like(h_col, device="cuda")
    d_val = torch.empty_like(h_val, device="cuda")
    Ad = binding.DeviceCSR(A.n_rows, A.n_cols, d_rp, d_col, d_val)
    copy_streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    parts = max(1, args.e2e_parts)

    def step():
        d_rp.copy_(h_rp, non_blocking=True)
        d_col.copy_(h_col, non_blocking=True)
        d_val.copy_(h_val, non_blocking=True)
        bounds = binding.gm_spgemm_row_split(Ad, Ad, parts, cfg, stream) if parts > 1 else [0, A.n_rows]
        held, base = [], 0
        for q in range(parts):
            r0, r1 = int(bounds[q]), int(bounds[q + 1])
            C = binding.spgemm(Ad, Ad, cfg, stream, rows=(r0, r1))
            binding.gm_row_ptr_shift(C.row_ptr, base, stream)
            ready = torch.cuda.Event()
            ready.record(stream)
            n = C.nnz
            cut = [0, n // 2, n]
            for k, cs in enumerate(copy_streams):
                cs.wait_event(ready)
                with torch.cuda.stream(cs):
                    if k == 0:
                        o_rp[r0:r1 + 1].copy_(C.row_ptr, non_blocking=True)
                    o_col[base + cut[k]:base + cut[k + 1]].copy_(C.col[cut[k]:cut[k + 1]], non_blocking=True)
                    o_val[base + cut[k]:base + cut[k + 1]].copy_(C.val[cut[k]:cut[k + 1]], non_blocking=True)
            held.append(C)  # alive until its copies are done
            base += n
        torch.cuda.synchronize()
        assert base == nnz_c
        held.clear()

    step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        step()
    dt = (time.perf_counter() - t0) / args.e2e_steps
    # context: the raw device-to-host rate of one large copy into the same pinned memory
    probe = min(nnz_c, 1 << 30)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    o_val[:probe].copy_(torch.empty(probe, dtype=o_val.dtype, device="cuda"), non_blocking=True)
    torch.cuda.synchronize()
    raw = probe * o_val.element_size() / (time.perf_counter() - t1) / 1e9
    return {"value": round(2.0 * ip_total / dt / 1e9, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(dt * 1e3, 2), "steps": args.e2e_steps,
            "parts": parts, "out_gbs_effective": round(d2h / dt / 1e9, 1), "raw_d2h_gbs": round(raw, 1),
            "pinned_on_gpu_numa_node": bool(cpus)}


def run_reference(args):
    """The CPU oracle, as it stands, on bounded row samples of the same workload."""
    import numpy as np

    import oracle
    from sparse_gemm_irregular_gm_gb300 import inputs
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    oracle.build()
    A, B = inputs.named_pair(args.workload, seed=args.seed)
    u = oracle.ip_counts(A, B)
    per_step = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    rng = np.random.default_rng(args.seed)
    order = rng.permutation(A.n_rows)
    csum = np.cumsum(u[order])
    k = min(A.n_rows, int(np.searchsorted(csum, 2e7)) + 1)
    t0 = time.perf_counter()
    oracle.spgemm_rows(A, B, np.sort(order[:k]))
    rate = float(csum[k - 1]) / max(time.perf_counter() - t0, 1e-3)
    k = min(A.n_rows, int(np.searchsorted(csum, rate * per_step)) + 1)
    rows = np.sort(order[:k])
    ip = int(csum[k - 1])
    for _ in range(args.warmup):
        oracle.spgemm_rows(A, B, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.spgemm_rows(A, B, rows)
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * ip / dt / 1e9
    sample = f"{k} random rows per step ({ip:.3e} of {int(u.sum()):.3e} intermediate products)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "A*A, A = R-MAT scale 20, edge factor 16, a=.57 b=.19 c=.19, fp64 U[-1,1), seed 1"
                   if args.workload == "rmat20" else args.workload, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.grid:
        run_grid(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
