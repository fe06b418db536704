"""C-ABI behaviour on the GPU: argument errors, host-buffer runs, the
format copy held on the device, and the bounded-wait failure detection."""
import numpy as np
import pytest

import oracle
import spmm_workloads as W
from spmm_testlib import ensure_library, run_library, to_device_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()
    import sparse_dense_matrix_bcsr_gb300 as S
    return S


def small(fmt, S):
    rng = np.random.default_rng(0)
    rp, ci, vals = W.random_csr(rng, 200, 300, 0.05, "bf16")
    if fmt == "bcsr":
        h = S.spmm_bcsr_create(200, 300, rp, ci, vals, "bf16", "f32")
    elif fmt == "wcsr":
        h = S.spmm_wcsr_create(200, 300, rp, ci, vals, "bf16", "f32")
    else:
        h = S.spmm_wcsr_create(200, 300, rp, ci, vals, "bf16", "f32", 64, 8)
    return h, rp, ci, vals


@pytest.mark.parametrize("fmt", ["bcsr", "wcsr"])
def test_run_argument_errors(S, fmt):
    import torch
    h, *_ = small(fmt, S)
    try:
        B = torch.zeros(300, 64, dtype=torch.bfloat16, device="cuda")
        C = torch.zeros(200, 64, dtype=torch.float32, device="cuda")
        assert S.spmm_run_status(h, B.data_ptr(), C.data_ptr(), 60, 0) == S.SPMM_ERR_UNSUPPORTED   # N % 8
        assert S.spmm_run_status(h, B.data_ptr() + 2, C.data_ptr(), 64, 0) == S.SPMM_ERR_UNSUPPORTED  # misaligned
        assert S.spmm_run_status(h, 0, C.data_ptr(), 64, 0) == S.SPMM_ERR_INVALID_ARG
        assert S.spmm_run_status(h, B.data_ptr(), C.data_ptr(), 0, 0) == S.SPMM_ERR_INVALID_ARG
        assert S.spmm_run_status(h, B.data_ptr(), C.data_ptr(), 64, 0) == S.SPMM_OK
        torch.cuda.synchronize()
        assert S.spmm_check(h, 0) == S.SPMM_OK
    finally:
        S.spmm_destroy(h)


@pytest.mark.parametrize("fmt", ["bcsr", "wcsr", "wcsr64"])
def test_device_format_matches_oracle(S, fmt):
    h, rp, ci, vals = small(fmt, S)
    try:
        got = S.spmm_export_format(h)
    finally:
        S.spmm_destroy(h)
    if fmt == "bcsr":
        ref = oracle.bcsr_build(200, 300, rp, ci, vals, 64, 64)
    elif fmt == "wcsr":
        ref = oracle.wcsr_build(200, 300, rp, ci, vals, 16, 16)
    else:
        ref = oracle.wcsr_build(200, 300, rp, ci, vals, 64, 8)
    for x, y in zip(ref, got):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("fmt", ["bcsr", "wcsr"])
def test_run_host_matches_run(S, fmt):
    rng = np.random.default_rng(1)
    m, k, n = 260, 333, 136
    rp, ci, vals = W.random_csr(rng, m, k, 0.04, "bf16")
    B = W.dense_bits(rng, (k, n), "n1", "bf16")
    outs, _ = run_library(fmt, m, k, rp, ci, vals, "bf16", "f32", B)
    h = (S.spmm_bcsr_create if fmt == "bcsr" else S.spmm_wcsr_create)(m, k, rp, ci, vals, "bf16", "f32")
    try:
        C = np.full((m, n), np.nan, np.float32)
        S.spmm_run_host(h, np.ascontiguousarray(B), C, n)
    finally:
        S.spmm_destroy(h)
    assert np.array_equal(C.astype(np.float64), outs[0])


@pytest.mark.parametrize("fmt,out_dt", [("bcsr", "bf16"), ("wcsr", "f32")])
def test_run_host_wide(S, fmt, out_dt):
    """spmm_run_host at N = 4104 (several column tiles and a ragged last one),
    called twice so the second call reuses the handle's staging buffers."""
    import oracle
    from spmm_testlib import assert_parity, ocode
    rng = np.random.default_rng(2)
    m, k, n = 260, 333, 4104
    rp, ci, vals = W.random_csr(rng, m, k, 0.04, "bf16")
    B = W.dense_bits(rng, (k, n), "n1", "bf16")
    outs, _ = run_library(fmt, m, k, rp, ci, vals, "bf16", out_dt, B)
    h = (S.spmm_bcsr_create if fmt == "bcsr" else S.spmm_wcsr_create)(m, k, rp, ci, vals, "bf16", out_dt)
    try:
        if out_dt == "f32":
            C = np.full((m, n), np.nan, np.float32)
        else:
            C = np.full((m, n), 0xFFFF, np.uint16)  # bf16 NaN bits
        for _ in range(2):
            S.spmm_run_host(h, np.ascontiguousarray(B), C, n)
    finally:
        S.spmm_destroy(h)
    Cd = C.astype(np.float64) if out_dt == "f32" else (C.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode("bf16"), B)
    assert_parity(Cd, C_ref, S_ref, f"{fmt} run_host N={n}")
    if fmt == "bcsr":  # same blocks in the same order per tile: bitwise equal to the device-buffer run
        assert np.array_equal(Cd, outs[0])


def test_bounded_wait_reports_timeout(S):
    """A wait that nothing completes ends after its limit with a recorded
    timeout; the context stays usable afterwards."""
    import torch
    assert S.spmm_selftest_wait_timeout(2_000_000) == S.SPMM_ERR_TIMEOUT
    x = torch.ones(4, device="cuda")
    assert float(x.sum().item()) == 4.0


def test_l2_read_probe_runs_and_leaves_sink(S):
    """The L2 read probe (the measured ceiling of the WCSR gather) reads its
    buffer without writing the sink and reports a plausible positive rate."""
    import torch
    buf = torch.ones(1 << 20, dtype=torch.int32, device="cuda")
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    S.spmm_probe_l2_read(buf.data_ptr(), buf.numel() * 4, 3, sink.data_ptr(), s.cuda_stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    S.spmm_probe_l2_read(buf.data_ptr(), buf.numel() * 4, 10, sink.data_ptr(), s.cuda_stream)
    e1.record(s)
    torch.cuda.synchronize()
    assert sink.abs().sum().item() == 0
    assert e0.elapsed_time(e1) > 0
