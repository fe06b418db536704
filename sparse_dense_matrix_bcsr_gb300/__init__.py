"""Python binding of the GB300 SpMM library (``include/spmm.h``).

Argument marshalling only: every step of the product runs in the CUDA
kernels of ``libspmm_gb300.so``.  The functions keep the C names:

    h = spmm_bcsr_create(m, k, row_ptr, col_idx, vals, in_t, out_t, b_row=64, b_col=64)
    h = spmm_wcsr_create(m, k, row_ptr, col_idx, vals, in_t, out_t, window_h=16, col_pad=16)
    spmm_run(h, B_ptr, C_ptr, N, stream_ptr)
    spmm_destroy(h)

plus ``spmm_format_info``, ``spmm_export_format``, ``spmm_check``,
``spmm_set_max_ctas``, ``spmm_run_host``, the host-only converters
``spmm_bcsr_convert`` / ``spmm_wcsr_convert`` and
``spmm_selftest_wait_timeout``.  ``run_torch`` is a convenience that passes
torch tensors and the current stream.

There is no fallback: if the shared library cannot be loaded, importing a
function that needs it raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspmm_gb300.so")

SPMM_OK = 0
SPMM_ERR_INVALID_ARG = 1
SPMM_ERR_UNSUPPORTED = 2
SPMM_ERR_CUDA = 3
SPMM_ERR_OOM = 4
SPMM_ERR_TIMEOUT = 5
SPMM_ERR_DEVICE_CHECK = 6

SPMM_F16 = 0
SPMM_BF16 = 1
SPMM_F32 = 2
DTYPES = {"f16": SPMM_F16, "bf16": SPMM_BF16, "f32": SPMM_F32}

SPMM_FORMAT_BCSR = 0
SPMM_FORMAT_WCSR = 1

# Every symbol the header declares.
EXPORTS = (
    "spmm_bcsr_create", "spmm_wcsr_create", "spmm_run", "spmm_run_host", "spmm_destroy",
    "spmm_format_info", "spmm_export_format", "spmm_bcsr_convert", "spmm_wcsr_convert",
    "spmm_check", "spmm_set_max_ctas", "spmm_selftest_wait_timeout", "spmm_status_str",
    "spmm_last_error", "spmm_wcsr_run_noalloc", "spmm_run_linear", "spmm_set_schedule",
    "spmm_probe_l2_read", "spmm_wcsr_noalloc_check",
)


class SpmmError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {_status_name(status)}: {msg}")
        self.status = status


class spmm_info(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int32), ("b_row", ctypes.c_int32), ("b_col", ctypes.c_int32),
        ("m", ctypes.c_int64), ("k", ctypes.c_int64), ("nnz", ctypes.c_int64),
        ("n_groups", ctypes.c_int64), ("n_units", ctypes.c_int64), ("stored", ctypes.c_int64),
        ("padding", ctypes.c_int64), ("idx_bytes", ctypes.c_int64), ("val_bytes", ctypes.c_int64),
        ("n_tasks", ctypes.c_int64), ("n_split_windows", ctypes.c_int64), ("split_cols", ctypes.c_int64),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libspmm_gb300.so (raises OSError if it is missing: build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing; build it with sparse_dense_matrix_bcsr_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I32 = ctypes.c_int
    st = ctypes.c_int
    sig = {
        "spmm_bcsr_create": [ctypes.POINTER(P), I64, I64, P, P, P, I32, I32, I32, I32],
        "spmm_wcsr_create": [ctypes.POINTER(P), I64, I64, P, P, P, I32, I32, I32, I32],
        "spmm_run": [P, P, P, I64, P],
        "spmm_run_linear": [P, P, P, I64, P],
        "spmm_run_host": [P, P, P, I64, P],
        "spmm_destroy": [P],
        "spmm_format_info": [P, ctypes.POINTER(spmm_info)],
        "spmm_export_format": [P, P, P, P],
        "spmm_bcsr_convert": [I64, I64, P, P, P, I32, I32, ctypes.POINTER(I64), P, P, P],
        "spmm_wcsr_convert": [I64, I64, P, P, P, I32, I32, ctypes.POINTER(I64), P, P, P],
        "spmm_check": [P, P],
        "spmm_set_max_ctas": [P, ctypes.c_int32],
        "spmm_set_schedule": [P, ctypes.c_int32],
        "spmm_selftest_wait_timeout": [I64, P, ctypes.POINTER(ctypes.c_int32)],
        "spmm_probe_l2_read": [P, I64, I32, P, P],
        "spmm_wcsr_noalloc_check": [P],
        "spmm_wcsr_run_noalloc": [P, P, P, I64, I64, I64, I32, I32, P, P, I64, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = st
    lib.spmm_status_str.argtypes = [st]
    lib.spmm_status_str.restype = ctypes.c_char_p
    lib.spmm_last_error.argtypes = []
    lib.spmm_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _status_name(s: int) -> str:
    try:
        return load_library().spmm_status_str(s).decode()
    except OSError:
        return str(s)


def _check(status: int, where: str):
    if status != SPMM_OK:
        msg = load_library().spmm_last_error().decode()
        raise SpmmError(status, where, msg)


def _arr(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _dt(t) -> int:
    return DTYPES[t] if isinstance(t, str) else int(t)


def _csr_args(row_ptr, col_idx, vals):
    rp, prp = _arr(row_ptr, np.int64)
    ci, pci = _arr(col_idx if len(col_idx) else np.zeros(1, np.int32), np.int32)
    vv, pvv = _arr(vals if len(vals) else np.zeros(1, np.uint16), np.uint16)
    return (rp, ci, vv), prp, pci, pvv


def spmm_bcsr_create(m, k, row_ptr, col_idx, vals, in_t="bf16", out_t="f32", b_row=64, b_col=64) -> int:
    lib = load_library()
    keep, prp, pci, pvv = _csr_args(row_ptr, col_idx, vals)
    h = ctypes.c_void_p()
    _check(lib.spmm_bcsr_create(ctypes.byref(h), m, k, prp, pci, pvv, _dt(in_t), _dt(out_t), b_row, b_col),
           "spmm_bcsr_create")
    return h.value


def spmm_wcsr_create(m, k, row_ptr, col_idx, vals, in_t="bf16", out_t="f32", window_h=16, col_pad=16) -> int:
    lib = load_library()
    keep, prp, pci, pvv = _csr_args(row_ptr, col_idx, vals)
    h = ctypes.c_void_p()
    _check(lib.spmm_wcsr_create(ctypes.byref(h), m, k, prp, pci, pvv, _dt(in_t), _dt(out_t), window_h, col_pad),
           "spmm_wcsr_create")
    return h.value


def spmm_run(h: int, B_ptr: int, C_ptr: int, N: int, stream: int = 0) -> None:
    _check(load_library().spmm_run(h, B_ptr, C_ptr, N, stream or None), "spmm_run")


def spmm_run_linear(h: int, X_ptr: int, Y_ptr: int, N: int, stream: int = 0) -> None:
    """Y = X * A^T on the GPU (BCSR handle; X is N x k, Y is N x m, both row-major device pointers)."""
    _check(load_library().spmm_run_linear(h, X_ptr, Y_ptr, N, stream or None), "spmm_run_linear")


def spmm_run_status(h: int, B_ptr: int, C_ptr: int, N: int, stream: int = 0) -> int:
    """spmm_run returning the raw status instead of raising."""
    return load_library().spmm_run(h, B_ptr, C_ptr, N, stream or None)


def spmm_run_host(h: int, B_host: np.ndarray, C_host: np.ndarray, N: int, stream: int = 0) -> None:
    assert B_host.flags.c_contiguous and C_host.flags.c_contiguous
    _check(load_library().spmm_run_host(h, B_host.ctypes.data, C_host.ctypes.data, N, stream or None),
           "spmm_run_host")


def spmm_run_host_ptr(h: int, B_ptr: int, C_ptr: int, N: int, stream: int = 0) -> None:
    _check(load_library().spmm_run_host(h, B_ptr, C_ptr, N, stream or None), "spmm_run_host")


def spmm_destroy(h: int) -> None:
    _check(load_library().spmm_destroy(h), "spmm_destroy")


def spmm_format_info(h: int) -> dict:
    info = spmm_info()
    _check(load_library().spmm_format_info(h, ctypes.byref(info)), "spmm_format_info")
    return {name: getattr(info, name) for name, _ in spmm_info._fields_}


def spmm_export_format(h: int):
    """(ptr int64, idx int32, vals uint16) host copies of the device format arrays."""
    info = spmm_format_info(h)
    ptr = np.zeros(info["n_groups"] + 1, np.int64)
    idx = np.zeros(max(info["n_units"], 1), np.int32)
    vals = np.zeros(max(info["stored"], 1), np.uint16)
    _check(load_library().spmm_export_format(h, ptr.ctypes.data, idx.ctypes.data, vals.ctypes.data),
           "spmm_export_format")
    idx = idx[: info["n_units"]]
    vals = vals[: info["stored"]]
    if info["format"] == SPMM_FORMAT_BCSR:
        vals = vals.reshape(info["n_units"], info["b_row"], info["b_col"])
    else:
        vals = vals.reshape(info["b_row"], info["n_units"])
    return ptr, idx, vals


def spmm_check(h: int, stream: int = 0) -> int:
    """Status word of the handle's kernels (SPMM_OK, SPMM_ERR_TIMEOUT, ...); does not raise."""
    return load_library().spmm_check(h, stream or None)


def spmm_set_max_ctas(h: int, ctas: int) -> None:
    _check(load_library().spmm_set_max_ctas(h, ctas), "spmm_set_max_ctas")


SPMM_SCHEDULE_AUTO = 0
SPMM_SCHEDULE_TILES = 1
SPMM_SCHEDULE_SPLIT = 2
SPMM_SCHEDULE_DYNAMIC = 3


def spmm_set_schedule(h: int, schedule: int) -> None:
    """Work schedule: SPMM_SCHEDULE_AUTO, _TILES, _SPLIT (BCSR) or _DYNAMIC (WCSR, window height 16)."""
    _check(load_library().spmm_set_schedule(h, schedule), "spmm_set_schedule")


def spmm_selftest_wait_timeout(timeout_ns: int, stream: int = 0) -> int:
    out = ctypes.c_int32(-1)
    _check(load_library().spmm_selftest_wait_timeout(timeout_ns, stream or None, ctypes.byref(out)),
           "spmm_selftest_wait_timeout")
    return out.value


def spmm_wcsr_noalloc_check(stream: int = 0) -> int:
    """Status of the last spmm_wcsr_run_noalloc call on the current device
    (waits for `stream`): SPMM_OK, SPMM_ERR_DEVICE_CHECK or SPMM_ERR_TIMEOUT."""
    return load_library().spmm_wcsr_noalloc_check(stream or None)


def spmm_probe_l2_read(buf: int, nbytes: int, passes: int, sink: int, stream: int = 0) -> None:
    """Enqueue `passes` reads of nbytes at device pointer buf (measurement helper)."""
    _check(load_library().spmm_probe_l2_read(buf, nbytes, passes, sink, stream or None), "spmm_probe_l2_read")


def spmm_wcsr_run_noalloc(window_row_ptr: int, window_col_idx: int, values: int, m: int, k: int, p_total: int,
                          in_t, out_t, B_ptr: int, C_ptr: int, N: int, stream: int = 0) -> None:
    """WCSR product from caller-owned device arrays, allocating nothing (pointers are device addresses)."""
    _check(load_library().spmm_wcsr_run_noalloc(window_row_ptr, window_col_idx, values, m, k, p_total, _dt(in_t),
                                                _dt(out_t), B_ptr, C_ptr, N, stream or None), "spmm_wcsr_run_noalloc")


def spmm_bcsr_convert(m, k, row_ptr, col_idx, vals, b_row=64, b_col=64):
    """Host-only CSR -> BCSR with the library's converter: (block_row_ptr, block_col_idx, blocks)."""
    lib = load_library()
    keep, prp, pci, pvv = _csr_args(row_ptr, col_idx, vals)
    nb = ctypes.c_int64(0)
    _check(lib.spmm_bcsr_convert(m, k, prp, pci, pvv, b_row, b_col, ctypes.byref(nb), None, None, None),
           "spmm_bcsr_convert")
    n = nb.value
    ptr = np.zeros(-(-m // b_row) + 1, np.int64)
    idx = np.zeros(max(n, 1), np.int32)
    blocks = np.zeros(max(n, 1) * b_row * b_col, np.uint16)
    _check(lib.spmm_bcsr_convert(m, k, prp, pci, pvv, b_row, b_col, ctypes.byref(nb), ptr.ctypes.data,
                                 idx.ctypes.data, blocks.ctypes.data), "spmm_bcsr_convert")
    return ptr, idx[:n], blocks[: n * b_row * b_col].reshape(n, b_row, b_col)


def spmm_wcsr_convert(m, k, row_ptr, col_idx, vals, window_h=16, col_pad=16):
    """Host-only CSR -> WCSR with the library's converter: (window_row_ptr, window_col_idx, values[h, P])."""
    lib = load_library()
    keep, prp, pci, pvv = _csr_args(row_ptr, col_idx, vals)
    pt = ctypes.c_int64(0)
    _check(lib.spmm_wcsr_convert(m, k, prp, pci, pvv, window_h, col_pad, ctypes.byref(pt), None, None, None),
           "spmm_wcsr_convert")
    P = pt.value
    ptr = np.zeros(-(-m // window_h) + 1, np.int64)
    idx = np.zeros(max(P, 1), np.int32)
    values = np.zeros(max(P, 1) * window_h, np.uint16)
    _check(lib.spmm_wcsr_convert(m, k, prp, pci, pvv, window_h, col_pad, ctypes.byref(pt), ptr.ctypes.data,
                                 idx.ctypes.data, values.ctypes.data), "spmm_wcsr_convert")
    return ptr, idx[:P], values[: P * window_h].reshape(window_h, P)


# ---------------------------------------------------------------- torch glue
def _torch_stream_ptr():
    import torch
    return torch.cuda.current_stream().cuda_stream


def run_torch(h: int, B, C, stream=None) -> None:
    """spmm_run on torch CUDA tensors B (k x N) and C (m x N), on the current stream."""
    assert B.is_cuda and C.is_cuda and B.is_contiguous() and C.is_contiguous()
    N = B.shape[1]
    assert C.shape[1] == N
    s = stream.cuda_stream if stream is not None else _torch_stream_ptr()
    spmm_run(h, B.data_ptr(), C.data_ptr(), N, s)


class SpMM:
    """Owning wrapper of one handle (destroyed with the object)."""

    def __init__(self, fmt: str, m: int, k: int, row_ptr, col_idx, vals, in_t="bf16", out_t="f32",
                 b_row=None, b_col=None):
        self.fmt = fmt
        self.m, self.k = m, k
        self.in_t, self.out_t = in_t, out_t
        if fmt == "bcsr":
            self.h = spmm_bcsr_create(m, k, row_ptr, col_idx, vals, in_t, out_t, b_row or 64, b_col or 64)
        elif fmt == "wcsr":
            self.h = spmm_wcsr_create(m, k, row_ptr, col_idx, vals, in_t, out_t, b_row or 16, b_col or 16)
        else:
            raise ValueError(fmt)

    def info(self) -> dict:
        return spmm_format_info(self.h)

    def __call__(self, B, C, stream=None):
        run_torch(self.h, B, C, stream)
        return C

    def check(self, stream: int = 0) -> int:
        return spmm_check(self.h, stream)

    def close(self):
        if getattr(self, "h", None):
            spmm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
