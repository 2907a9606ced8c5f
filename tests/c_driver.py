"""Builds and feeds tests/c_abi_driver.c, a plain C program that calls the C ABI.

Test infrastructure only: binary CSR files in the driver's layout (int64 n_rows,
n_cols, nnz; int64 row_ptr; int32 col; float64 val, little endian).
"""
import os
import shutil
import subprocess

import numpy as np

from sparse_gemm_irregular_gm_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB_DIR = os.path.join(ROOT, "sparse_gemm_irregular_gm_gb300")


def cuda_home() -> str:
    return os.environ.get("CUDA_HOME") or "/usr/local/cuda"


def build_c_driver(out_dir: str) -> str:
    """Compile and link the driver with the host C compiler against
    libgm_spgemm.so and the CUDA runtime; returns the executable's path."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler")
    exe = os.path.join(out_dir, "c_abi_driver")
    cuda_lib = os.path.join(cuda_home(), "lib64")
    subprocess.run([cc, "-std=c11", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda_home(), "include"), os.path.join(HERE, "c_abi_driver.c"),
                    "-o", exe, "-L", LIB_DIR, "-lgm_spgemm", "-L", cuda_lib, "-lcudart",
                    f"-Wl,-rpath,{LIB_DIR}", f"-Wl,-rpath,{cuda_lib}"], check=True)
    return exe


def write_csr(path: str, M) -> None:
    with open(path, "wb") as f:
        np.array([M.n_rows, M.n_cols, M.nnz], dtype="<i8").tofile(f)
        M.row_ptr.astype("<i8").tofile(f)
        M.col.astype("<i4").tofile(f)
        M.val.astype("<f8").tofile(f)


def read_csr(path: str):
    with open(path, "rb") as f:
        n_rows, n_cols, nnz = (int(x) for x in np.fromfile(f, dtype="<i8", count=3))
        rp = np.fromfile(f, dtype="<i8", count=n_rows + 1).astype(np.int64)
        col = np.fromfile(f, dtype="<i4", count=nnz).astype(np.int32)
        val = np.fromfile(f, dtype="<f8", count=nnz).astype(np.float64)
    return inputs.CSR(n_rows, n_cols, rp, col, val)
