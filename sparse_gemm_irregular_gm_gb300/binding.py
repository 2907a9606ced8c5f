"""ctypes binding of libgm_spgemm.so (include/gm_spgemm.h), same names as the C ABI.

Argument marshalling only: every step of the SpGEMM runs in the CUDA library.
torch supplies device memory and the stream. There is no CPU fallback: when the
library is missing or cannot load, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
# GM_SPGEMM_CHECKED=1 selects the GM_BOUNDS_CHECK build of the library (build.py)
LIB_PATH = os.path.join(HERE, "libgm_spgemm_checked.so" if os.environ.get("GM_SPGEMM_CHECKED") == "1"
                        else "libgm_spgemm.so")

GM_MAX_LEVELS = 16
GM_NUM_STAGES = 16
STATUS_NAMES = ["GM_OK", "GM_ERR_INVALID_ARG", "GM_ERR_DIM_MISMATCH", "GM_ERR_INDEX_OVERFLOW", "GM_ERR_OOM",
                "GM_ERR_WORKSPACE", "GM_ERR_CUDA", "GM_ERR_DEVICE_TIMEOUT", "GM_ERR_STATE", "GM_ERR_BAD_INDEX",
                "GM_ERR_INTERNAL"]
GM_FLAG_TIMING, GM_FLAG_KEEP_INTERMEDIATES, GM_FLAG_LOG, GM_FLAG_OVERLAP = 1, 2, 4, 8
GM_VALUE_F64, GM_VALUE_F32 = 0, 1
GM_INDEX_ROWPTR32, GM_INDEX_COL64 = 1, 2
GM_PIPE_AUTO, GM_PIPE_UNFUSED, GM_PIPE_FUSED_HISTO, GM_PIPE_ROWWISE = 0, 1, 2, 3
PIPELINES = {GM_PIPE_AUTO: "auto", GM_PIPE_UNFUSED: "outer-product, unfused",
             GM_PIPE_FUSED_HISTO: "outer-product, fused level-0 histogram",
             GM_PIPE_ROWWISE: "direct to level-0 chunks (C-hat not written)"}
(GM_DBG_IP_COUNTS, GM_DBG_HEAVY_ROWS, GM_DBG_LIGHT_ROWS, GM_DBG_CHAT_ROWPTR, GM_DBG_CHAT_COL, GM_DBG_CHAT_VAL,
 GM_DBG_REORD_ROWPTR, GM_DBG_REORD_COL, GM_DBG_REORD_VAL, GM_DBG_REORD_CHILD) = range(10)
STAGES = ["analyze", "transpose", "outer", "histogram", "multisplit", "sym_heavy", "sym_light", "scan",
          "num_heavy", "num_light", "other", "transpose_sym", "outer_sym", "histogram_sym", "multisplit_sym",
          "unused"]
EXPORTS = ["gm_set_allocator", "gm_spgemm_params", "gm_spgemm_analyze", "gm_spgemm_symbolic", "gm_spgemm_numeric",
           "gm_spgemm_plan_info", "gm_spgemm_plan_destroy", "gm_status_string", "gm_spgemm_debug_copy",
           "gm_prefix_sum_noalloc", "gm_spgemm_analyze_rows", "gm_spgemm_row_split", "gm_row_ptr_shift"]


class gm_csr(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int64), ("n_cols", ctypes.c_int64), ("nnz", ctypes.c_int64),
                ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p), ("vals", ctypes.c_void_p)]


class gm_config(ctypes.Structure):
    _fields_ = [("smem_budget_bytes", ctypes.c_int64), ("tau", ctypes.c_int64), ("dense_width", ctypes.c_int64),
                ("n_chunks_max", ctypes.c_int64), ("workspace_cap_bytes", ctypes.c_int64),
                ("pipeline", ctypes.c_int32), ("flags", ctypes.c_int32), ("value_type", ctypes.c_int32),
                ("index_type", ctypes.c_int32)]


class gm_params(ctypes.Structure):
    _fields_ = [("s_lm", ctypes.c_int64), ("tau", ctypes.c_int64), ("dense_width", ctypes.c_int64),
                ("n_chunks_required", ctypes.c_int64), ("n_chunks_max", ctypes.c_int64),
                ("n_levels", ctypes.c_int64), ("v_chunks", ctypes.c_int64 * GM_MAX_LEVELS),
                ("widths", ctypes.c_int64 * GM_MAX_LEVELS)]


class gm_plan_info(ctypes.Structure):
    _fields_ = [("params", gm_params), ("n_rows", ctypes.c_int64), ("n_cols", ctypes.c_int64),
                ("n_heavy_rows", ctypes.c_int64), ("n_light_rows", ctypes.c_int64),
                ("n_empty_rows", ctypes.c_int64), ("ip_total", ctypes.c_int64), ("ip_heavy", ctypes.c_int64),
                ("c_nnz", ctypes.c_int64), ("chat_bytes", ctypes.c_int64), ("n_batches", ctypes.c_int64),
                ("workspace_peak_bytes", ctypes.c_int64), ("n_leaves", ctypes.c_int64),
                ("keeps_reordered", ctypes.c_int32), ("pipeline", ctypes.c_int32),
                ("cuda_error", ctypes.c_int32), ("device_status", ctypes.c_int32),
                ("stage_ms", ctypes.c_float * GM_NUM_STAGES), ("kernel_launches", ctypes.c_int64),
                ("value_type", ctypes.c_int32), ("chunk_col_bytes", ctypes.c_int32),
                ("index_type", ctypes.c_int32)]


class GmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{where}: {name}")


_lib = None


def load(path: str = LIB_PATH):
    """Load libgm_spgemm.so (built by ``build.build()``); raises when it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.gm_set_allocator.restype = None
    lib.gm_set_allocator.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.gm_spgemm_params.restype = ctypes.c_int
    lib.gm_spgemm_params.argtypes = [ctypes.c_int64, P(gm_config), P(gm_params)]
    lib.gm_spgemm_analyze.restype = ctypes.c_int
    lib.gm_spgemm_analyze.argtypes = [P(gm_csr), P(gm_csr), P(gm_config), ctypes.c_void_p, P(ctypes.c_void_p)]
    lib.gm_spgemm_symbolic.restype = ctypes.c_int
    lib.gm_spgemm_symbolic.argtypes = [ctypes.c_void_p, ctypes.c_void_p, P(ctypes.c_int64)]
    lib.gm_spgemm_numeric.restype = ctypes.c_int
    lib.gm_spgemm_numeric.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.gm_spgemm_plan_info.restype = ctypes.c_int
    lib.gm_spgemm_plan_info.argtypes = [ctypes.c_void_p, P(gm_plan_info)]
    lib.gm_spgemm_plan_destroy.restype = None
    lib.gm_spgemm_plan_destroy.argtypes = [ctypes.c_void_p]
    lib.gm_status_string.restype = ctypes.c_char_p
    lib.gm_status_string.argtypes = [ctypes.c_int]
    lib.gm_spgemm_debug_copy.restype = ctypes.c_int
    lib.gm_spgemm_debug_copy.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_int64, P(ctypes.c_int64)]
    lib.gm_spgemm_analyze_rows.restype = ctypes.c_int
    lib.gm_spgemm_analyze_rows.argtypes = [P(gm_csr), P(gm_csr), ctypes.c_int64, ctypes.c_int64, P(gm_config),
                                           ctypes.c_void_p, P(ctypes.c_void_p)]
    lib.gm_spgemm_row_split.restype = ctypes.c_int
    lib.gm_spgemm_row_split.argtypes = [P(gm_csr), P(gm_csr), P(gm_config), ctypes.c_int64, ctypes.c_void_p,
                                        P(ctypes.c_int64)]
    lib.gm_row_ptr_shift.restype = ctypes.c_int
    lib.gm_row_ptr_shift.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                     ctypes.c_void_p]
    lib.gm_prefix_sum_noalloc.restype = ctypes.c_int
    lib.gm_prefix_sum_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                          ctypes.c_void_p]
    _lib = lib
    use_torch_allocator(True)
    return lib


# ---- workspace through torch's caching allocator ---------------------------------
# The plan's workspace (up to hundreds of GB for large products) is taken from and
# returned to torch's cache, so repeated products reuse the same device memory
# instead of mapping and unmapping it each time.
_ALLOC_T = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
_FREE_T = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
_AVAIL_T = ctypes.CFUNCTYPE(ctypes.c_int64, ctypes.c_void_p)
_hooks = None


def _torch_alloc(ctx, nbytes, stream):
    import torch
    for attempt in range(2):
        try:
            return torch.cuda.caching_allocator_alloc(int(nbytes), torch.cuda.current_device(), stream or 0)
        except Exception:
            if attempt == 0:
                torch.cuda.empty_cache()
    return None


def _torch_free(ctx, ptr, nbytes, stream):
    import torch
    torch.cuda.caching_allocator_delete(ptr)


def _torch_avail(ctx):
    import torch
    try:
        free, _ = torch.cuda.mem_get_info()
        return int(free + torch.cuda.memory_reserved() - torch.cuda.memory_allocated())
    except Exception:
        return -1


def use_torch_allocator(enable: bool = True):
    """Route workspace allocations through torch (enable) or back to cudaMallocAsync."""
    global _hooks
    lib = _lib
    if lib is None:
        return
    if enable:
        try:
            import torch
            if not torch.cuda.is_available():
                return
        except ImportError:
            return
        _hooks = (_ALLOC_T(_torch_alloc), _FREE_T(_torch_free), _AVAIL_T(_torch_avail))
        lib.gm_set_allocator(ctypes.cast(_hooks[0], ctypes.c_void_p), ctypes.cast(_hooks[1], ctypes.c_void_p),
                             ctypes.cast(_hooks[2], ctypes.c_void_p), None)
    else:
        lib.gm_set_allocator(None, None, None, None)
        _hooks = None


def _check(rc: int, where: str):
    if rc != 0:
        raise GmError(rc, where)


def make_config(**kw) -> gm_config:
    cfg = gm_config()
    for k, v in kw.items():
        setattr(cfg, k, int(v))
    return cfg


def gm_status_string(status: int) -> str:
    return load().gm_status_string(status).decode()


def gm_spgemm_params(c_m: int, cfg: gm_config | None = None) -> gm_params:
    out = gm_params()
    _check(load().gm_spgemm_params(int(c_m), ctypes.byref(cfg) if cfg else None, ctypes.byref(out)),
           "gm_spgemm_params")
    return out


@dataclass
class DeviceCSR:
    """CSR operand whose arrays are torch CUDA tensors: row pointers int64 or int32, columns int32 or
    int64, values float64 or float32."""

    n_rows: int
    n_cols: int
    row_ptr: object
    col: object
    val: object

    @property
    def nnz(self) -> int:
        return int(self.col.numel())

    def desc(self) -> gm_csr:
        return gm_csr(self.n_rows, self.n_cols, self.nnz, self.row_ptr.data_ptr(),
                      self.col.data_ptr() if self.nnz else None, self.val.data_ptr() if self.nnz else None)


def to_device(M, device="cuda", dtype=None, row_ptr_dtype=None, col_dtype=None) -> DeviceCSR:
    """Copy a host CSR (``inputs.CSR``) to torch CUDA tensors; values as ``dtype``
    (numpy float32 or float64), row pointers as ``row_ptr_dtype`` (int64 or
    int32), columns as ``col_dtype`` (int32 or int64); default: as stored."""
    import torch
    val = M.val if dtype is None else M.val.astype(dtype)
    rp = M.row_ptr if row_ptr_dtype is None else M.row_ptr.astype(row_ptr_dtype)
    col = M.col if col_dtype is None else M.col.astype(col_dtype)
    return DeviceCSR(M.n_rows, M.n_cols, torch.from_numpy(rp).to(device),
                     torch.from_numpy(col).to(device), torch.from_numpy(val).to(device))


def _value_type(A: DeviceCSR, B: DeviceCSR) -> int:
    """GM_VALUE_* of the operands' value tensors (A and B must agree)."""
    import torch
    kinds = {torch.float64: GM_VALUE_F64, torch.float32: GM_VALUE_F32}
    ta, tb = kinds.get(A.val.dtype), kinds.get(B.val.dtype)
    if ta is None or tb is None or ta != tb:
        raise GmError(1, f"values must be float64 or float32 in both A and B, not {A.val.dtype} and {B.val.dtype}")
    return ta


def _index_type(A: DeviceCSR, B: DeviceCSR) -> int:
    """GM_INDEX_* flags of the operands' row-pointer and column tensors (A and B must agree)."""
    import torch
    rp = {torch.int64: 0, torch.int32: GM_INDEX_ROWPTR32}
    col = {torch.int32: 0, torch.int64: GM_INDEX_COL64}
    ra, rb = rp.get(A.row_ptr.dtype), rp.get(B.row_ptr.dtype)
    ca, cb = col.get(A.col.dtype), col.get(B.col.dtype)
    if ra is None or ra != rb:
        raise GmError(1, f"row pointers must be int64 or int32 in both A and B, not {A.row_ptr.dtype} and "
                         f"{B.row_ptr.dtype}")
    if ca is None or ca != cb:
        raise GmError(1, f"columns must be int32 or int64 in both A and B, not {A.col.dtype} and {B.col.dtype}")
    return ra | ca


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _typed_config(A: DeviceCSR, B: DeviceCSR, cfg: gm_config | None):
    """cfg (or None) with value_type and index_type taken from the operands' tensor dtypes."""
    vt = _value_type(A, B)
    it = _index_type(A, B)
    if cfg is None and (vt != GM_VALUE_F64 or it != 0):
        cfg = gm_config()
    if cfg is not None:
        cfg = gm_config.from_buffer_copy(cfg)
        cfg.value_type = vt
        cfg.index_type = it
    return cfg


def gm_spgemm_analyze(A: DeviceCSR, B: DeviceCSR, cfg: gm_config | None = None, stream=None, rows=None):
    """gm_spgemm_analyze (or, with rows = (row_begin, row_end), gm_spgemm_analyze_rows)
    with cfg.value_type and cfg.index_type taken from the operands' tensor dtypes."""
    plan = ctypes.c_void_p()
    a, b = A.desc(), B.desc()
    cfg = _typed_config(A, B, cfg)
    c = ctypes.byref(cfg) if cfg else None
    if rows is None:
        _check(load().gm_spgemm_analyze(ctypes.byref(a), ctypes.byref(b), c, _stream_handle(stream),
                                        ctypes.byref(plan)), "gm_spgemm_analyze")
    else:
        _check(load().gm_spgemm_analyze_rows(ctypes.byref(a), ctypes.byref(b), int(rows[0]), int(rows[1]), c,
                                             _stream_handle(stream), ctypes.byref(plan)), "gm_spgemm_analyze_rows")
    return plan


def gm_spgemm_row_split(A: DeviceCSR, B: DeviceCSR, n_parts: int, cfg: gm_config | None = None, stream=None):
    """Row bounds (numpy int64, n_parts + 1) of a split of A's rows into parts of about equal products."""
    import numpy as np
    a, b = A.desc(), B.desc()
    cfg = _typed_config(A, B, cfg)
    out = np.zeros(int(n_parts) + 1, dtype=np.int64)
    _check(load().gm_spgemm_row_split(ctypes.byref(a), ctypes.byref(b), ctypes.byref(cfg) if cfg else None,
                                      int(n_parts), _stream_handle(stream),
                                      out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))), "gm_spgemm_row_split")
    return out


def gm_row_ptr_shift(row_ptr, base: int, stream=None):
    """Adds base to every entry of a CUDA row-pointer tensor (int64 or int32), in place."""
    import torch
    if row_ptr.dtype not in (torch.int64, torch.int32) or not row_ptr.is_contiguous() or not row_ptr.is_cuda:
        raise ValueError("row_ptr must be a contiguous int64 or int32 CUDA tensor")
    it = GM_INDEX_ROWPTR32 if row_ptr.dtype == torch.int32 else 0
    _check(load().gm_row_ptr_shift(row_ptr.data_ptr() if row_ptr.numel() else None, row_ptr.numel(), int(base),
                                   it, _stream_handle(stream)), "gm_row_ptr_shift")


def gm_spgemm_symbolic(plan, c_row_ptr) -> int:
    nnz = ctypes.c_int64(-1)
    _check(load().gm_spgemm_symbolic(plan, c_row_ptr.data_ptr(), ctypes.byref(nnz)), "gm_spgemm_symbolic")
    return int(nnz.value)


def gm_spgemm_numeric(plan, c_col, c_val):
    _check(load().gm_spgemm_numeric(plan, c_col.data_ptr() if c_col.numel() else None,
                                    c_val.data_ptr() if c_val.numel() else None), "gm_spgemm_numeric")


def gm_spgemm_plan_info(plan) -> gm_plan_info:
    out = gm_plan_info()
    _check(load().gm_spgemm_plan_info(plan, ctypes.byref(out)), "gm_spgemm_plan_info")
    return out


def gm_spgemm_plan_destroy(plan):
    load().gm_spgemm_plan_destroy(plan)


def gm_spgemm_debug_copy(plan, view: int, level: int = 0):
    """Host numpy copy of a plan array (see the GM_DBG_* views of the header)."""
    import numpy as np
    size = ctypes.c_int64(0)
    _check(load().gm_spgemm_debug_copy(plan, view, level, None, 0, ctypes.byref(size)), "gm_spgemm_debug_copy")
    vdt = np.float32 if gm_spgemm_plan_info(plan).value_type == GM_VALUE_F32 else np.float64
    dtype = {GM_DBG_HEAVY_ROWS: np.int32, GM_DBG_LIGHT_ROWS: np.int32, GM_DBG_CHAT_COL: np.int32,
             GM_DBG_REORD_COL: np.int32, GM_DBG_CHAT_VAL: vdt, GM_DBG_REORD_VAL: vdt}.get(view, np.int64)
    out = np.empty(size.value // np.dtype(dtype).itemsize, dtype=dtype)
    if size.value:
        _check(load().gm_spgemm_debug_copy(plan, view, level, out.ctypes.data, size.value, None),
               "gm_spgemm_debug_copy")
    return out


def gm_prefix_sum_noalloc(inp, out, total=None, stream=None):
    """Exclusive scan of an int64 CUDA tensor into ``out`` using the library's fixed scratch.

    ``inp`` and ``out`` are contiguous int64 tensors on the current CUDA device,
    ``out`` at least as long as ``inp`` (it may be ``inp`` itself); ``total``, when
    given, a contiguous int64 tensor of at least one element on the same device.
    Anything else raises ValueError before the library is called."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    named = [("inp", inp), ("out", out)] + ([("total", total)] if total is not None else [])
    for name, t in named:
        if not isinstance(t, torch.Tensor) or t.dtype != torch.int64 or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"{name} must be a contiguous int64 tensor on {dev}")
    if out.numel() < inp.numel():
        raise ValueError(f"out holds {out.numel()} elements, the scan writes {inp.numel()}")
    if total is not None and total.numel() < 1:
        raise ValueError("total must hold at least one element")
    _check(load().gm_prefix_sum_noalloc(inp.data_ptr() if inp.numel() else None,
                                        out.data_ptr() if out.numel() else None, inp.numel(),
                                        total.data_ptr() if total is not None else None,
                                        _stream_handle(stream)), "gm_prefix_sum_noalloc")


def spgemm(A: DeviceCSR, B: DeviceCSR, cfg: gm_config | None = None, stream=None, return_info: bool = False,
           rows=None):
    """C = A @ B on the GPU: analyze, symbolic, allocate C with torch, numeric.
    With rows = (row_begin, row_end): those rows of C only (row pointers from 0)."""
    import torch
    dev = A.row_ptr.device
    plan = gm_spgemm_analyze(A, B, cfg, stream, rows=rows)
    n_out = A.n_rows if rows is None else int(rows[1]) - int(rows[0])
    try:
        c_rp = torch.empty(n_out + 1, dtype=A.row_ptr.dtype, device=dev)
        nnz = gm_spgemm_symbolic(plan, c_rp)
        c_col = torch.empty(nnz, dtype=A.col.dtype, device=dev)
        c_val = torch.empty(nnz, dtype=A.val.dtype, device=dev)
        gm_spgemm_numeric(plan, c_col, c_val)
        info = gm_spgemm_plan_info(plan) if return_info else None
    finally:
        gm_spgemm_plan_destroy(plan)
    C = DeviceCSR(n_out, B.n_cols, c_rp, c_col, c_val)
    return (C, info) if return_info else C
