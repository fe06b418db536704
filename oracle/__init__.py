"""CPU oracle for sparse x dense SpMM and the BCSR / WCSR formats.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the library under ``sparse_dense_matrix_bcsr_gb300/``.

Everything is computed by ``oracle.c`` (plain C, fp64 accumulation), compiled
with gcc into ``liboracle.so`` next to this file; this module only marshals
numpy arrays.  The formats follow "AsyncSparse: Accelerating Sparse
Matrix-Matrix Multiplication on Asynchronous GPU Architectures", Section II-C
and Fig. 2; the SpMM follows its problem statement C = A x B.

Parity status of each function (what pins it, see tests/test_oracle_pins.py):
  csr_check        pinned: hand-made invalid CSRs.
  bcsr_build       pinned: Fig. 2 index arrays; brute-force block enumeration
                   from a dense copy; stored = nnz + padding; fill ratio.
  wcsr_build       pinned: Fig. 2 index arrays; brute-force column unions from
                   a dense copy; stored = nnz + padding.
  spmm_csr         pinned: dense fp64 matmul (numpy) of the densified matrix;
                   identity and one-nonzero-per-row closed forms.
  spmm_csr_sample  pinned: equals spmm_csr at the sampled positions.
  spmm_bcsr/wcsr   pinned: equal spmm_csr (block-diagonal / window cases too).
  half decoding    pinned: numpy float16 and the bfloat16 bit definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F16 = 0
BF16 = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (OpenMP on)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.orc_half_to_double.restype = ctypes.c_double
    lib.orc_half_to_double.argtypes = [ctypes.c_uint16, i32]
    lib.orc_csr_check.restype = i32
    lib.orc_csr_check.argtypes = [i64, i64, p, p]
    lib.orc_bcsr_nblocks.restype = i64
    lib.orc_bcsr_nblocks.argtypes = [i64, i64, p, p, i32, i32]
    lib.orc_bcsr_build.restype = None
    lib.orc_bcsr_build.argtypes = [i64, i64, p, p, p, i32, i32, p, p, p]
    lib.orc_wcsr_ncols.restype = i64
    lib.orc_wcsr_ncols.argtypes = [i64, i64, p, p, i32, i32]
    lib.orc_wcsr_build.restype = None
    lib.orc_wcsr_build.argtypes = [i64, i64, p, p, p, i32, i32, p, p, p]
    lib.orc_spmm_csr.restype = None
    lib.orc_spmm_csr.argtypes = [i64, i64, i64, p, p, p, i32, p, p, p, i32]
    lib.orc_spmm_csr_sample.restype = None
    lib.orc_spmm_csr_sample.argtypes = [i64, i64, i64, p, p, p, i32, p, i64, p, p, p, p]
    lib.orc_spmm_bcsr.restype = None
    lib.orc_spmm_bcsr.argtypes = [i64, i64, i64, i32, i32, p, p, p, i32, p, p]
    lib.orc_spmm_wcsr.restype = None
    lib.orc_spmm_wcsr.argtypes = [i64, i64, i64, i32, p, p, p, i32, p, p]
    lib.orc_num_threads.restype = i32
    lib.orc_num_threads.argtypes = []
    _lib = lib
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _csr(row_ptr, col_idx, vals=None):
    rp = _c(row_ptr, np.int64)
    ci = _c(col_idx, np.int32)
    if vals is None:
        return rp, ci
    return rp, ci, _c(vals, np.uint16)


def half_to_double(bits: int, dtype: int) -> float:
    return _load().orc_half_to_double(int(bits), int(dtype))


def csr_check(m: int, k: int, row_ptr, col_idx) -> int:
    """0 if the CSR is valid; 1 bad row_ptr, 2 column out of range, 3 unsorted/duplicate."""
    rp, ci = _csr(row_ptr, col_idx)
    if len(rp) != m + 1 or (m >= 0 and len(ci) < rp[-1]):
        return 1
    if len(ci) == 0:
        ci = np.zeros(1, np.int32)
    return _load().orc_csr_check(m, k, _ptr(rp), _ptr(ci))


def bcsr_build(m: int, k: int, row_ptr, col_idx, vals, b_row: int = 64, b_col: int = 64):
    """CSR -> BCSR.  Returns (block_row_ptr int64, block_col_idx int32, blocks uint16 [nb, b_row, b_col])."""
    lib = _load()
    rp, ci, v = _csr(row_ptr, col_idx, vals)
    ci_ = ci if len(ci) else np.zeros(1, np.int32)
    v_ = v if len(v) else np.zeros(1, np.uint16)
    nb = lib.orc_bcsr_nblocks(m, k, _ptr(rp), _ptr(ci_), b_row, b_col)
    nbr = -(-m // b_row)
    brp = np.zeros(nbr + 1, np.int64)
    bci = np.zeros(max(nb, 1), np.int32)
    blocks = np.zeros(max(nb, 1) * b_row * b_col, np.uint16)
    lib.orc_bcsr_build(m, k, _ptr(rp), _ptr(ci_), _ptr(v_), b_row, b_col, _ptr(brp), _ptr(bci), _ptr(blocks))
    return brp, bci[:nb], blocks[: nb * b_row * b_col].reshape(nb, b_row, b_col)


def wcsr_build(m: int, k: int, row_ptr, col_idx, vals, h: int = 16, pad: int = 16):
    """CSR -> WCSR.  Returns (window_row_ptr int64, window_col_idx int32, values uint16 [h, P_total])."""
    lib = _load()
    rp, ci, v = _csr(row_ptr, col_idx, vals)
    ci_ = ci if len(ci) else np.zeros(1, np.int32)
    v_ = v if len(v) else np.zeros(1, np.uint16)
    P = lib.orc_wcsr_ncols(m, k, _ptr(rp), _ptr(ci_), h, pad)
    nw = -(-m // h)
    wrp = np.zeros(nw + 1, np.int64)
    wci = np.zeros(max(P, 1), np.int32)
    values = np.zeros(max(P, 1) * h, np.uint16)
    lib.orc_wcsr_build(m, k, _ptr(rp), _ptr(ci_), _ptr(v_), h, pad, _ptr(wrp), _ptr(wci), _ptr(values))
    if P == 0:
        return wrp, wci[:0], np.zeros((h, 0), np.uint16)
    return wrp, wci[:P], values.reshape(h, P)


def spmm_csr(m: int, k: int, row_ptr, col_idx, vals, dtype: int, B, threads: int = 0, with_abs: bool = True):
    """fp64 C = A*B from the CSR, and S = sum |a*b| (None if with_abs is False)."""
    lib = _load()
    rp, ci, v = _csr(row_ptr, col_idx, vals)
    ci_ = ci if len(ci) else np.zeros(1, np.int32)
    v_ = v if len(v) else np.zeros(1, np.uint16)
    Bb = _c(B, np.uint16)
    n = Bb.shape[1]
    C = np.empty((m, n), np.float64)
    S = np.empty((m, n), np.float64) if with_abs else None
    lib.orc_spmm_csr(m, k, n, _ptr(rp), _ptr(ci_), _ptr(v_), dtype, _ptr(Bb), _ptr(C),
                     _ptr(S) if S is not None else None, threads)
    return C, S


def spmm_csr_sample(m: int, k: int, row_ptr, col_idx, vals, dtype: int, B, rows, cols):
    """fp64 C[rows[t], cols[t]] and S at the same positions."""
    lib = _load()
    rp, ci, v = _csr(row_ptr, col_idx, vals)
    ci_ = ci if len(ci) else np.zeros(1, np.int32)
    v_ = v if len(v) else np.zeros(1, np.uint16)
    Bb = B if (isinstance(B, np.ndarray) and B.dtype == np.uint16 and B.flags.c_contiguous) else _c(B, np.uint16)
    n = Bb.shape[1]
    r = _c(rows, np.int64)
    c = _c(cols, np.int64)
    C = np.empty(len(r), np.float64)
    S = np.empty(len(r), np.float64)
    lib.orc_spmm_csr_sample(m, k, n, _ptr(rp), _ptr(ci_), _ptr(v_), dtype, _ptr(Bb), len(r),
                            _ptr(r), _ptr(c), _ptr(C), _ptr(S))
    return C, S


def spmm_bcsr(m: int, k: int, block_row_ptr, block_col_idx, blocks, dtype: int, B):
    lib = _load()
    blocks = _c(blocks, np.uint16)
    b_row, b_col = blocks.shape[1], blocks.shape[2]
    brp = _c(block_row_ptr, np.int64)
    bci = _c(block_col_idx, np.int32)
    bci_ = bci if len(bci) else np.zeros(1, np.int32)
    bl_ = blocks.reshape(-1) if blocks.size else np.zeros(1, np.uint16)
    Bb = _c(B, np.uint16)
    n = Bb.shape[1]
    C = np.empty((m, n), np.float64)
    lib.orc_spmm_bcsr(m, k, n, b_row, b_col, _ptr(brp), _ptr(bci_), _ptr(bl_), dtype, _ptr(Bb), _ptr(C))
    return C


def spmm_wcsr(m: int, k: int, window_row_ptr, window_col_idx, values, dtype: int, B):
    lib = _load()
    values = _c(values, np.uint16)
    h = values.shape[0]
    wrp = _c(window_row_ptr, np.int64)
    wci = _c(window_col_idx, np.int32)
    wci_ = wci if len(wci) else np.zeros(1, np.int32)
    v_ = values.reshape(-1) if values.size else np.zeros(1, np.uint16)
    Bb = _c(B, np.uint16)
    n = Bb.shape[1]
    C = np.empty((m, n), np.float64)
    lib.orc_spmm_wcsr(m, k, n, h, _ptr(wrp), _ptr(wci_), _ptr(v_), dtype, _ptr(Bb), _ptr(C))
    return C


def num_threads() -> int:
    return _load().orc_num_threads()


def within_tolerance(C_gpu, C_ref, S_ref):
    """Per-element bound |C_gpu - C_ref| <= 4 * 2^-8 * S + 1e-6 (bf16/fp16 inputs, fp32 accumulation).

    Returns (ok, worst_ratio) where worst_ratio = max |err| / bound."""
    C_gpu = np.asarray(C_gpu, np.float64)
    err = np.abs(C_gpu - C_ref)
    bound = 4.0 * 2.0 ** -8 * S_ref + 1e-6
    bad = ~(err <= bound)  # NaN counts as a failure
    ratio = float(np.nanmax(err / bound)) if err.size else 0.0
    if np.isnan(C_gpu).any():
        ratio = float("inf")
    return (not bad.any()), ratio
