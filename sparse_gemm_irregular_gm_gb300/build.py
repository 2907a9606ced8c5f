"""Builds libgm_spgemm.so (CUDA, sm_103a) in-tree with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then one
nvcc call links the shared library. Objects go to ``_build/`` next to this file.
``build(checked=True)`` builds libgm_spgemm_checked.so instead, with
GM_BOUNDS_CHECK defined: every write of C and of the chunk elements checks its
index first and reports an index out of range as GM_ERR_INTERNAL (objects in
``_build_checked/``). The binding loads it when GM_SPGEMM_CHECKED=1.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgm_spgemm.so")
LIB_CHECKED = os.path.join(HERE, "libgm_spgemm_checked.so")
SOURCES = ["gm_api.cu", "gm_analyze.cu", "gm_scan.cu", "gm_expand.cu", "gm_multisplit.cu", "gm_accum.cu", "gm_rowbitmap.cu",
           "gm_stream.cu", "gm_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "gm_spgemm.h")]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile (if stale) and return the path of libgm_spgemm.so (or, with checked,
    of libgm_spgemm_checked.so)."""
    lib = LIB_CHECKED if checked else LIB
    bdir = BUILD + "_checked" if checked else BUILD
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}"]
    if checked:
        flags.append("-DGM_BOUNDS_CHECK")

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-ldl",  # NVTX loads a profiler's hooks
           "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
