"""Host-side checks of the C ABI that need no GPU.

The library loads, exports every function include/gm_spgemm.h declares, its
parameter selection equals the oracle's (gMAGNUS Sec. III-D) including the
51 chunk counts of Tables V/VI, and argument errors are caught on the host.
"""
import ctypes
import json
import os
import re

import pytest

import oracle
from sparse_gemm_irregular_gm_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return binding.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gm_spgemm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\**\s*(gm_[a-z_]+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(binding.EXPORTS) == names


def test_status_strings(lib):
    for i, name in enumerate(binding.STATUS_NAMES):
        assert binding.gm_status_string(i).startswith(name)


def _lib_params(c_m, **kw):
    return binding.gm_spgemm_params(c_m, binding.make_config(**kw) if kw else None)


@pytest.mark.parametrize("c_m", [1, 2, 8, 1000, 1 << 10, (1 << 14) + 1, 1 << 18, 1 << 20, (1 << 21) + 7, 10 ** 8])
@pytest.mark.parametrize("over", [{}, {"tau": 64, "dense_width": 64, "n_chunks_max": 4},
                                  {"dense_width": 256, "n_chunks_max": 2}, {"smem_budget_bytes": 65536},
                                  {"smem_budget_bytes": 49152, "tau": 100, "n_chunks_max": 8}])
def test_params_match_oracle(lib, c_m, over):
    kw = {}
    if "smem_budget_bytes" in over:
        kw["s_lm"] = over["smem_budget_bytes"]
    for k in ("tau", "dense_width", "n_chunks_max"):
        if k in over:
            kw[k] = over[k]
    ref = oracle.magnus_params(c_m, **kw)
    if ref.n_levels > binding.GM_MAX_LEVELS:  # the ABI holds at most 16 levels
        with pytest.raises(binding.GmError) as e:
            _lib_params(c_m, **over)
        assert e.value.status == 3
        return
    got = _lib_params(c_m, **over)
    assert got.s_lm == ref.s_lm and got.tau == ref.tau
    assert got.dense_width == ref.dense_width and got.n_chunks_max == ref.n_chunks_max
    assert got.n_chunks_required == ref.n_chunks_required and got.n_levels == ref.n_levels
    assert list(got.v_chunks[:got.n_levels]) == ref.v_chunks
    assert list(got.widths[:got.n_levels]) == ref.widths


@pytest.mark.parametrize("c_m", [1, 1000, (1 << 14) + 1, 1 << 18, 1 << 20, (1 << 21) + 7, 10 ** 8])
@pytest.mark.parametrize("over", [{}, {"tau": 64, "dense_width": 64, "n_chunks_max": 4}, {"smem_budget_bytes": 65536}])
def test_params_float_values_match_oracle(lib, c_m, over):
    """The planner with 4-byte values (gm_config.value_type = GM_VALUE_F32) is
    GetMagnusParams with s_C.val = 4: at 227 KB tau = 232448 / (2 * 8) = 14528 and
    the dense width floor_pow2(232448 / 5) = 32768, twice the double one."""
    kw = {"s_lm": over["smem_budget_bytes"]} if "smem_budget_bytes" in over else {}
    kw.update({k: over[k] for k in ("tau", "dense_width", "n_chunks_max") if k in over})
    ref = oracle.magnus_params(c_m, s_val=4, **kw)
    if ref.n_levels > binding.GM_MAX_LEVELS:
        return
    got = _lib_params(c_m, value_type=binding.GM_VALUE_F32, **over)
    assert (got.tau, got.dense_width, got.n_chunks_max) == (ref.tau, ref.dense_width, ref.n_chunks_max)
    assert got.n_chunks_required == ref.n_chunks_required and got.n_levels == ref.n_levels
    assert list(got.v_chunks[:got.n_levels]) == ref.v_chunks
    assert list(got.widths[:got.n_levels]) == ref.widths
    if not over:
        assert (got.tau, got.dense_width) == (14528, 32768)
        dbl = _lib_params(c_m)
        assert (dbl.tau, dbl.dense_width) == (9685, 16384)


def test_params_float_rejects_what_the_oracle_rejects(lib):
    """With 4-byte values and tau = 16, Eq. (6) leaves no room for a histogram
    (n_chunksMax < 1): the oracle raises and the library returns an error."""
    with pytest.raises(ValueError):
        oracle.magnus_params(1024, s_val=4, tau=16)
    with pytest.raises(binding.GmError) as e:
        _lib_params(1024, tau=16, value_type=binding.GM_VALUE_F32)
    assert e.value.status == 1
    assert _lib_params(1024, tau=32, value_type=binding.GM_VALUE_F32).n_levels == 0


def test_params_rejects_unknown_value_type(lib):
    with pytest.raises(binding.GmError) as e:
        _lib_params(1 << 20, value_type=7)
    assert e.value.status == 1


def test_params_tables_v_vi(lib):
    with open(os.path.join(ROOT, "tests", "golden", "magnus_chunk_tables.json")) as f:
        g = json.load(f)
    n = 0
    for row in g["suitesparse"] + [[f"rmat{s}", 1 << s, p, h] for s, p, h in g["rmat"]]:
        _, c_m, pvc, h200 = row
        for gpu, entry in (("PVC", pvc), ("H200", h200)):
            if entry is None:
                continue
            cal = g["calibration"][gpu]
            p = _lib_params(c_m, dense_width=cal["dense_width"], n_chunks_max=cal["n_chunks_max"])
            req = int(entry.split(":")[0])
            levels = [int(x) for x in entry.split(":")[1].split(",")] if ":" in entry else [req]
            assert p.n_chunks_required == req
            assert list(p.v_chunks[:p.n_levels]) == levels
            n += 1
    assert n == 51


def test_params_rejects_bad_overrides(lib):
    for kw in ({"dense_width": 100}, {"n_chunks_max": 3}, {"n_chunks_max": 1}, {"tau": 10 ** 6},
               {"smem_budget_bytes": 10 ** 7}):
        with pytest.raises(binding.GmError) as e:
            _lib_params(1 << 20, **kw)
        assert e.value.status == 1
    with pytest.raises(binding.GmError):
        _lib_params(0)


def test_analyze_host_argument_errors(lib):
    fake = 0x1000  # never dereferenced: every check below fails on the host
    A = binding.gm_csr(4, 5, 3, fake, fake, fake)
    B = binding.gm_csr(6, 5, 3, fake, fake, fake)
    plan = ctypes.c_void_p()
    assert lib.gm_spgemm_analyze(ctypes.byref(A), ctypes.byref(B), None, None, ctypes.byref(plan)) == 2
    B.n_rows = 5
    assert lib.gm_spgemm_analyze(None, ctypes.byref(B), None, None, ctypes.byref(plan)) == 1
    assert lib.gm_spgemm_analyze(ctypes.byref(A), ctypes.byref(B), None, None, None) == 1
    bad = binding.gm_csr(-1, 5, 3, fake, fake, fake)
    assert lib.gm_spgemm_analyze(ctypes.byref(bad), ctypes.byref(B), None, None, ctypes.byref(plan)) == 1
    nul = binding.gm_csr(4, 5, 3, fake, None, fake)
    assert lib.gm_spgemm_analyze(ctypes.byref(nul), ctypes.byref(B), None, None, ctypes.byref(plan)) == 1
    big = binding.gm_csr(1 << 31, 5, 3, fake, fake, fake)
    assert lib.gm_spgemm_analyze(ctypes.byref(big), ctypes.byref(B), None, None, ctypes.byref(plan)) == 3
    assert not plan.value


def test_plan_calls_reject_null(lib):
    assert lib.gm_spgemm_symbolic(None, None, None) == 1
    assert lib.gm_spgemm_numeric(None, None, None) == 1
    assert lib.gm_spgemm_plan_info(None, None) == 1
    lib.gm_spgemm_plan_destroy(None)


def test_params_no_level_needed_with_small_tau(lib):
    # tau = 16 leaves Eq. (6) a single chunk per level; fine while C.m <= D needs no level.
    got = _lib_params(1024, tau=16)
    ref = oracle.magnus_params(1024, tau=16)
    assert (got.n_chunks_max, got.n_levels) == (ref.n_chunks_max, ref.n_levels) == (1, 0)
    with pytest.raises(binding.GmError):
        _lib_params(1 << 20, tau=16)


def test_analyze_index_type_host_errors(lib):
    """Unknown index flags are rejected, and int32 row pointers cannot describe a
    matrix with 2^31 or more entries; both before any device work."""
    fake = 0x1000  # never dereferenced
    A = binding.gm_csr(4, 5, 3, fake, fake, fake)
    B = binding.gm_csr(5, 5, 3, fake, fake, fake)
    plan = ctypes.c_void_p()
    for flags in (4, 8, -1):
        cfg = binding.make_config(index_type=flags)
        assert lib.gm_spgemm_analyze(ctypes.byref(A), ctypes.byref(B), ctypes.byref(cfg), None,
                                     ctypes.byref(plan)) == 1
    big = binding.gm_csr(4, 5, 1 << 31, fake, fake, fake)
    cfg = binding.make_config(index_type=binding.GM_INDEX_ROWPTR32)
    assert lib.gm_spgemm_analyze(ctypes.byref(big), ctypes.byref(B), ctypes.byref(cfg), None,
                                 ctypes.byref(plan)) == 3
    assert lib.gm_spgemm_analyze(ctypes.byref(A), ctypes.byref(big), ctypes.byref(cfg), None,
                                 ctypes.byref(plan)) == 3
    assert not plan.value


def test_analyze_rejects_unknown_pipelines(lib):
    """gm_config.pipeline takes GM_PIPE_AUTO .. GM_PIPE_ROWWISE; any other value is
    an argument error found on the host."""
    fake = 0x1000  # never dereferenced
    A = binding.gm_csr(4, 5, 3, fake, fake, fake)
    B = binding.gm_csr(5, 5, 3, fake, fake, fake)
    plan = ctypes.c_void_p()
    for pipeline in (-1, 4, 99):
        cfg = binding.make_config(pipeline=pipeline)
        assert lib.gm_spgemm_analyze(ctypes.byref(A), ctypes.byref(B), ctypes.byref(cfg), None,
                                     ctypes.byref(plan)) == 1
    assert not plan.value


@pytest.mark.parametrize("c_m", [1 << 10, 1 << 20, 1 << 24])
def test_params_do_not_depend_on_index_type(lib, c_m):
    """The planner sizes shared memory by the widths held there (int32 columns,
    int64 row pointers), which the interface's index types do not change."""
    ref = _lib_params(c_m)
    for flags in (binding.GM_INDEX_ROWPTR32, binding.GM_INDEX_COL64, 3):
        got = _lib_params(c_m, index_type=flags)
        assert (got.tau, got.dense_width, got.n_chunks_max, got.n_levels) == \
               (ref.tau, ref.dense_width, ref.n_chunks_max, ref.n_levels)


def test_struct_layouts_match_the_header(tmp_path):
    """The binding's ctypes structures have the sizes and field offsets a C
    compiler gives the header's structs."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"gm_csr": binding.gm_csr, "gm_config": binding.gm_config, "gm_params": binding.gm_params,
               "gm_plan_info": binding.gm_plan_info}
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "gm_spgemm.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{name}.{field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                       text=True).stdout.splitlines())
    for name, cls in structs.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert int(got[f"{name}.{field}"]) == getattr(cls, field).offset, f"{name}.{field}"


def test_binding_index_type_from_dtypes():
    """The binding derives gm_config.index_type from the operands' tensor dtypes
    and refuses mixed or unsupported ones (host logic only)."""
    torch = pytest.importorskip("torch")

    def csr(rp_dt, col_dt):
        return binding.DeviceCSR(2, 2, torch.zeros(3, dtype=rp_dt), torch.zeros(0, dtype=col_dt),
                                 torch.zeros(0, dtype=torch.float64))

    i64, i32 = torch.int64, torch.int32
    assert binding._index_type(csr(i64, i32), csr(i64, i32)) == 0
    assert binding._index_type(csr(i32, i32), csr(i32, i32)) == binding.GM_INDEX_ROWPTR32
    assert binding._index_type(csr(i64, i64), csr(i64, i64)) == binding.GM_INDEX_COL64
    assert binding._index_type(csr(i32, i64), csr(i32, i64)) == binding.GM_INDEX_ROWPTR32 | binding.GM_INDEX_COL64
    for a, b in ((csr(i32, i32), csr(i64, i32)), (csr(i64, i64), csr(i64, i32)), (csr(torch.int16, i32),) * 2,
                 (csr(i64, torch.uint8),) * 2):
        with pytest.raises(binding.GmError):
            binding._index_type(a, b)


def test_c_program_compiles_and_links_against_the_library(lib, tmp_path):
    """A plain C program (tests/c_abi_driver.c) builds against include/gm_spgemm.h
    and links every call it makes from libgm_spgemm.so (running it needs a GPU:
    tests/test_gpu_parity.py::test_c_program_through_the_abi)."""
    from tests.c_driver import build_c_driver
    exe = build_c_driver(str(tmp_path))
    assert os.access(exe, os.X_OK)


def test_missing_library_fails_loudly(tmp_path):
    """Without the CUDA library the binding raises when it loads: there is no CPU
    fallback (run in a fresh interpreter, since a loaded library is cached)."""
    import subprocess
    import sys
    code = ("import sys\n"
            f"sys.path.insert(0, {ROOT!r})\n"
            "from sparse_gemm_irregular_gm_gb300 import binding\n"
            "try:\n"
            f"    binding.load({str(tmp_path / 'absent.so')!r})\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n"
            "    sys.exit(3)\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 3, r.stdout + r.stderr
    assert "missing" in r.stdout


def test_params_at_the_widest_products(lib):
    """C.m = 2^31 (the widest C the interface takes) gets the oracle's plan, three
    levels of 256, 256 and 2 chunks at 227 KB; the planner's chunk space ends at
    D * n_chunksRequired = 2^32 columns, beyond which it reports an overflow."""
    for c_m in (1 << 31, 1 << 32):
        got, ref = _lib_params(c_m), oracle.magnus_params(c_m)
        assert got.n_levels == ref.n_levels == 3
        assert list(got.v_chunks[:3]) == list(ref.v_chunks)
    assert list(_lib_params(1 << 31).v_chunks[:3]) == [256, 256, 2]
    for c_m in ((1 << 32) + 1, 1 << 40):
        with pytest.raises(binding.GmError) as e:
            _lib_params(c_m)
        assert e.value.status == 3
