"""C-ABI library on the host (no GPU): it loads, exports every symbol that
include/spmm.h declares, and its CSR -> BCSR / WCSR converters match the
oracle's bit for bit; invalid input is rejected."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import spmm_workloads as W
from spmm_testlib import ROOT, ensure_library


@pytest.fixture(scope="module")
def lib():
    ensure_library()
    import sparse_dense_matrix_bcsr_gb300 as S
    return S


def declared_functions():
    src = open(os.path.join(ROOT, "include", "spmm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spmm_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 14
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(so, n), n
    assert set(names) == set(lib.EXPORTS)


def test_status_strings(lib):
    L = lib.load_library()
    assert L.spmm_status_str(0) == b"SPMM_OK"
    assert L.spmm_status_str(5) == b"SPMM_ERR_TIMEOUT"


def test_fig2_through_library_converter(lib):
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "fig2_formats.json")))
    rp = np.cumsum([0] + [len(r) for r in g["rows"]]).astype(np.int64)
    ci = np.array(sum(g["rows"], []), np.int32)
    vals = W.f32_to_f16_bits(np.arange(1, len(ci) + 1, dtype=np.float32))
    p, i, _ = lib.spmm_bcsr_convert(g["m"], g["k"], rp, ci, vals, g["b_row"], g["b_col"])
    assert p.tolist() == g["expected"]["block_row_ptr"] and i.tolist() == g["expected"]["block_col_idx"]
    p, i, _ = lib.spmm_wcsr_convert(g["m"], g["k"], rp, ci, vals, g["b_row"], g["b_col"])
    assert p.tolist() == g["expected"]["window_row_ptr"] and i.tolist() == g["expected"]["window_col_idx"]


CASES = [
    (1, 1, 1.0, 64, 64), (100, 37, 0.05, 64, 64), (300, 500, 0.01, 64, 64), (64, 4096, 0.002, 64, 64),
    (257, 129, 0.2, 16, 16), (1000, 800, 0.003, 16, 16), (33, 1000, 0.05, 16, 32), (0, 10, 0.1, 16, 16),
    (50, 50, 0.0, 16, 16), (17, 19, 0.3, 4, 4), (129, 200, 0.1, 8, 16),
    (300, 700, 0.02, 64, 8), (1000, 1000, 0.01, 64, 8), (65, 129, 0.1, 64, 16),
]


@pytest.mark.parametrize("m,k,d,a,b", CASES)
def test_converters_bit_exact_vs_oracle(lib, m, k, d, a, b):
    rng = np.random.default_rng(1000 + m * 7 + k)
    rp, ci, vals = W.random_csr(rng, m, k, d, "bf16")
    ob = oracle.bcsr_build(m, k, rp, ci, vals, a, b)
    lb = lib.spmm_bcsr_convert(m, k, rp, ci, vals, a, b)
    for x, y in zip(ob, lb):
        assert x.dtype == y.dtype and np.array_equal(x, y)
    ow = oracle.wcsr_build(m, k, rp, ci, vals, a, b)
    lw = lib.spmm_wcsr_convert(m, k, rp, ci, vals, a, b)
    for x, y in zip(ow, lw):
        assert x.dtype == y.dtype and np.array_equal(x, y)


def test_converters_on_config_shapes(lib):
    """The BCSR tiny workload and a scaled-down power-law WCSR workload."""
    w = W.bcsr_tiny()
    for x, y in zip(oracle.bcsr_build(w.m, w.k, w.row_ptr, w.col_idx, w.vals, 64, 64),
                    lib.spmm_bcsr_convert(w.m, w.k, w.row_ptr, w.col_idx, w.vals, 64, 64)):
        assert np.array_equal(x, y)
    rng = np.random.default_rng(77)
    rp, ci = W.powerlaw_pattern(rng, 8192, 8192, 1.8, 1, 2000, 256, 0.7)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    for x, y in zip(oracle.wcsr_build(8192, 8192, rp, ci, vals, 16, 16),
                    lib.spmm_wcsr_convert(8192, 8192, rp, ci, vals, 16, 16)):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("rp,ci", [([1, 2, 3], [0, 3, 1]), ([0, 2, 1], [0, 3, 1]), ([0, 2, 3], [0, 4, 1]),
                                   ([0, 2, 3], [3, 0, 1]), ([0, 2, 3], [2, 2, 1]), ([0, 2, 3], [0, -1, 1])])
def test_invalid_csr_rejected(lib, rp, ci):
    vals = np.ones(3, np.uint16)
    with pytest.raises(lib.SpmmError) as e:
        lib.spmm_bcsr_convert(2, 4, np.array(rp), np.array(ci), vals, 64, 64)
    assert e.value.status == lib.SPMM_ERR_INVALID_ARG
    with pytest.raises(lib.SpmmError) as e:
        lib.spmm_wcsr_create(2, 4, np.array(rp), np.array(ci), vals)
    assert e.value.status == lib.SPMM_ERR_INVALID_ARG


def test_bad_parameters_rejected(lib):
    rp = np.array([0, 1], np.int64)
    ci = np.array([0], np.int32)
    v = np.ones(1, np.uint16)
    for args in [dict(b_row=0), dict(b_col=300)]:
        with pytest.raises(lib.SpmmError):
            lib.spmm_bcsr_convert(1, 1, rp, ci, v, **args)
    with pytest.raises(lib.SpmmError) as e:
        lib.spmm_bcsr_create(1, 1, rp, ci, v, "f32", "f32")
    assert e.value.status == lib.SPMM_ERR_INVALID_ARG
    with pytest.raises(lib.SpmmError) as e:
        lib.spmm_run(0, 16, 16, 8, 0)
    assert e.value.status == lib.SPMM_ERR_INVALID_ARG


def test_l2_probe_rejects_bad_arguments_before_any_device_call(lib):
    L = lib.load_library()
    sink = ctypes.c_void_p(16)
    assert L.spmm_probe_l2_read(None, 1024, 1, sink, None) == lib.SPMM_ERR_INVALID_ARG
    assert L.spmm_probe_l2_read(ctypes.c_void_p(16), 1000, 1, sink, None) == lib.SPMM_ERR_INVALID_ARG
    assert L.spmm_probe_l2_read(ctypes.c_void_p(16), 1024, 0, sink, None) == lib.SPMM_ERR_INVALID_ARG
    assert L.spmm_probe_l2_read(ctypes.c_void_p(8), 1024, 1, sink, None) == lib.SPMM_ERR_INVALID_ARG
