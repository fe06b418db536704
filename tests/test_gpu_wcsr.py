"""WCSR kernel (and its split-window reduction) parity with the oracle on
the GPU, through the C ABI."""
import numpy as np
import pytest

import oracle
import spmm_workloads as W
from spmm_testlib import (assert_parity, ensure_library, ocode, run_library, sampled_parity,
                          stratified_positions)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def full_check(m, k, n, rp, ci, vals, dt, out_dt, B, max_ctas=None, runs=1):
    outs, info = run_library("wcsr", m, k, rp, ci, vals, dt, out_dt, B, max_ctas=max_ctas, runs=runs)
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode(dt), B)
    for C in outs:
        assert_parity(C, C_ref, S_ref, f"wcsr {m}x{k} N={n}")
    return outs, info


@pytest.mark.parametrize("m,k,n,d,dt,out_dt", [
    (512, 512, 128, 0.05, "bf16", "f32"),
    (1000, 3000, 256, 0.01, "bf16", "f32"),
    (333, 777, 72, 0.03, "f16", "f32"),       # ragged window, N < 128
    (256, 2048, 264, 0.02, "bf16", "bf16"),   # two column tiles + tail, bf16 C
    (64, 64, 8, 0.2, "bf16", "f32"),          # N = 8
    (333, 777, 40, 0.03, "f16", "f32"),       # N <= 64, ragged window
    (1000, 3000, 64, 0.01, "bf16", "bf16"),   # N = 64, bf16 C
    (700, 4000, 24, 0.02, "bf16", "f32"),     # N = 24: partial 16-byte units
])
def test_wcsr_parity_small(m, k, n, d, dt, out_dt):
    rng = np.random.default_rng(m + 17 * n)
    rp, ci, vals = W.random_csr(rng, m, k, d, dt)
    B = W.dense_bits(rng, (k, n), "n1", dt)
    full_check(m, k, n, rp, ci, vals, dt, out_dt, B)


@pytest.mark.parametrize("ctas,n,out_dt", [(3, 256, "f32"), (7, 128, "f32"), (13, 72, "f32"), (5, 520, "f32"),
                                          (6, 264, "bf16"), (7, 64, "f32"), (11, 40, "bf16"), (4, 8, "f32")])
def test_wcsr_windows_cut_between_ctas(ctas, n, out_dt):
    """Few persistent CTAs: long windows are cut between CTAs and finished by
    the second kernel; the result must match and be bitwise reproducible."""
    rng = np.random.default_rng(ctas)
    m, k = 400, 5000
    rp, ci = W.powerlaw_pattern(rng, m, k, 1.3, 1, 1500, 300, 0.7)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    B = W.dense_bits(rng, (k, n), "u1", "bf16")
    outs, info = full_check(m, k, n, rp, ci, vals, "bf16", out_dt, B, max_ctas=ctas, runs=2)
    assert info["n_split_windows"] > 0
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("n", [136, 48])
def test_wcsr_window_spanning_many_ctas(n):
    """One window much longer than a CTA's share: its partials span several CTAs."""
    rng = np.random.default_rng(17)
    m, k = 48, 6000
    rp = np.zeros(m + 1, np.int64)
    cols = [np.sort(rng.choice(k, 3000 if i == 20 else 3, replace=False)) for i in range(m)]
    rp[1:] = np.cumsum([len(c) for c in cols])
    ci = np.concatenate(cols).astype(np.int32)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    B = W.dense_bits(rng, (k, n), "u1", "bf16")
    full_check(m, k, n, rp, ci, vals, "bf16", "bf16", B, max_ctas=9, runs=1)


def test_wcsr_empty_windows_and_identity():
    m = 300
    n = 24
    rp = np.arange(m + 1, dtype=np.int64)
    ci = np.arange(m, dtype=np.int32)
    one = W.f32_to_bf16_bits(np.ones(m, np.float32))
    # drop rows 32..95 (four windows) to get empty windows
    keep = np.ones(m, bool)
    keep[32:96] = False
    rows = np.nonzero(keep)[0]
    rp2 = np.zeros(m + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=m), out=rp2[1:])
    B = W.dense_bits(np.random.default_rng(2), (m, n), "n1", "bf16")
    outs, _ = run_library("wcsr", m, m, rp2, ci[keep], one[keep], "bf16", "f32", B)
    ref = W.bits_to_f32(B, "bf16").astype(np.float64)
    ref[32:96] = 0
    assert np.array_equal(outs[0], ref)


@pytest.mark.parametrize("n", [136, 56])
def test_wcsr_one_nonzero_per_row_exact(n):
    rng = np.random.default_rng(9)
    m, k = 257, 900
    rp = np.arange(m + 1, dtype=np.int64)
    ci = rng.integers(0, k, m).astype(np.int32)
    vals = W.draw_values(rng, m, "u1", "f16")
    B = W.dense_bits(rng, (k, n), "u1", "f16")
    outs, _ = run_library("wcsr", m, k, rp, ci, vals, "f16", "f32", B, max_ctas=5)
    ref = vals.view(np.float16).astype(np.float64)[:, None] * B.view(np.float16).astype(np.float64)[ci]
    assert np.array_equal(outs[0], ref)


def sampled_check(w, nsamp=8000, seed=0, max_ctas=None):
    """Full-size workload: C fully written (no NaN left), then one sampled
    output in every (window, 128-column strip) cell plus nsamp uniform ones
    compared with the oracle."""
    import torch
    outs, info = run_library("wcsr", w.m, w.k, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.B(),
                             keep_device=True, max_ctas=max_ctas)
    C = outs[0]
    assert not torch.isnan(C).any().item(), "C not fully written"
    rows, cols = stratified_positions(w.m, w.n, 16, nsamp, seed)
    sampled_parity(w, C, rows, cols)
    return info


def test_wcsr_uniform_full_size():
    w = W.wcsr_uniform()
    outs, info = full_check(w.m, w.k, w.n, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.B())
    assert info["n_groups"] == 1024


def test_wcsr_irregular_full_size():
    """The irregular workload at full size (262144 rows, N = 128), every
    element of C compared with the oracle."""
    w = W.wcsr_irregular()
    outs, info = full_check(w.m, w.k, w.n, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.B())
    assert info["n_split_windows"] > 0  # windows cut between CTAs


@pytest.mark.parametrize("dens", W.WCSR_SWEEP_DENSITY)
@pytest.mark.parametrize("n", W.SWEEP_N)
def test_wcsr_sweep_full_size_sampled(dens, n):
    sampled_check(W.wcsr_sweep(dens, n))


# ---------------------------------------------------------------- 64-row windows
@pytest.mark.parametrize("m,k,n,d,pad,out_dt,ctas", [
    (512, 512, 256, 0.05, 8, "f32", None),
    (1000, 3000, 256, 0.01, 8, "f32", None),
    (333, 777, 72, 0.03, 8, "f32", None),        # ragged window, N < 256: live columns only
    (256, 2048, 264, 0.02, 16, "bf16", None),    # two column tiles + tail, bf16 C
    (64, 64, 8, 0.2, 8, "f32", None),            # N = 8
    (400, 5000, 256, 0.02, 8, "f32", 3),         # few CTAs: windows cut between CTAs
    (400, 5000, 136, 0.02, 8, "bf16", 7),
])
def test_wcsr64_parity(m, k, n, d, pad, out_dt, ctas):
    """Windows of 64 rows with column padding 8 or 16 (the paper's WCSR
    configuration, Section IV-A), element by element against the oracle and
    bitwise reproducible."""
    rng = np.random.default_rng(m + 3 * n + pad)
    rp, ci, vals = W.random_csr(rng, m, k, d, "bf16")
    B = W.dense_bits(rng, (k, n), "n1", "bf16")
    outs, info = run_library("wcsr", m, k, rp, ci, vals, "bf16", out_dt, B, b_row=64, b_col=pad,
                             max_ctas=ctas, runs=2)
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode("bf16"), B)
    for C in outs:
        assert_parity(C, C_ref, S_ref, f"wcsr64 {m}x{k} N={n} pad={pad}")
    assert np.array_equal(outs[0], outs[1])
    if ctas:
        assert info["n_split_windows"] > 0


def test_wcsr64_long_window_over_many_ctas():
    rng = np.random.default_rng(23)
    m, k, n = 192, 6000, 264
    cols = [np.sort(rng.choice(k, 3000 if i == 70 else 5, replace=False)) for i in range(m)]
    rp = np.zeros(m + 1, np.int64)
    rp[1:] = np.cumsum([len(c) for c in cols])
    ci = np.concatenate(cols).astype(np.int32)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    B = W.dense_bits(rng, (k, n), "u1", "bf16")
    outs, _ = run_library("wcsr", m, k, rp, ci, vals, "bf16", "f32", B, b_row=64, b_col=8, max_ctas=11)
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode("bf16"), B)
    assert_parity(outs[0], C_ref, S_ref, "wcsr64 long window")


def test_wcsr64_identity_and_empty_windows_exact():
    m = 300
    n = 24
    keep = np.ones(m, bool)
    keep[64:192] = False  # two empty windows
    rows = np.nonzero(keep)[0]
    rp = np.zeros(m + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=m), out=rp[1:])
    ci = rows.astype(np.int32)
    one = W.f32_to_bf16_bits(np.ones(len(ci), np.float32))
    B = W.dense_bits(np.random.default_rng(2), (m, n), "n1", "bf16")
    outs, _ = run_library("wcsr", m, m, rp, ci, one, "bf16", "f32", B, b_row=64, b_col=8)
    ref = W.bits_to_f32(B, "bf16").astype(np.float64)
    ref[64:192] = 0
    assert np.array_equal(outs[0], ref)


def test_wcsr64_uniform_full_size():
    """The uniform workload (16384^2, 1 %, N = 256) in 64-row windows, every
    element compared with the oracle."""
    w = W.wcsr_uniform()
    outs, info = run_library("wcsr", w.m, w.k, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.B(),
                             b_row=64, b_col=8)
    C_ref, S_ref = oracle.spmm_csr(w.m, w.k, w.row_ptr, w.col_idx, w.vals, ocode(w.dtype), w.B())
    assert_parity(outs[0], C_ref, S_ref, "wcsr_uniform h64")
    assert info["n_groups"] == 256


def _dyn_run(w_or_args, max_ctas=None, runs=2):
    import sparse_dense_matrix_bcsr_gb300 as S
    m, k, n, rp, ci, vals, dt, out_dt, B = w_or_args
    return run_library("wcsr", m, k, rp, ci, vals, dt, out_dt, B, max_ctas=max_ctas, runs=runs,
                       schedule=S.SPMM_SCHEDULE_DYNAMIC)


def test_wcsr_dynamic_schedule_takes_over_chunks():
    """Dynamic schedule with more chunks than CTAs fit on the GPU (about four
    per resident CTA), so running CTAs cancel pending ones through cluster
    launch control and take their chunks: every element matches the oracle,
    and two runs are bitwise equal (the chunks are fixed and their partial
    sums are added in chunk order, whichever CTA ran them)."""
    rng = np.random.default_rng(2026)
    m, k, n = 20000, 20000, 128
    rp, ci, vals = W.random_csr(rng, m, k, 0.005, "bf16")
    B = W.dense_bits(rng, (k, n), "u1", "bf16")
    outs, info = _dyn_run((m, k, n, rp, ci, vals, "bf16", "f32", B))
    assert info["n_tasks"] >= 32 * 4 * 152, "too few work items to give every chunk 32"
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode("bf16"), B)
    for C in outs:
        assert_parity(C, C_ref, S_ref, "wcsr dynamic")
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("ctas,n,out_dt", [(3, 256, "f32"), (5, 72, "bf16"), (2, 520, "f32"), (4, 40, "f32")])
def test_wcsr_dynamic_schedule_few_chunks(ctas, n, out_dt):
    """Dynamic schedule with a CTA cap: a handful of chunks (all resident at
    once, so every cancellation request finds nothing left), long windows cut
    between chunks; parity with the oracle and bitwise-equal runs."""
    rng = np.random.default_rng(300 + ctas)
    m, k = 2400, 5000
    rp, ci = W.powerlaw_pattern(rng, m, k, 1.3, 1, 1500, 300, 0.7)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    B = W.dense_bits(rng, (k, n), "u1", "bf16")
    outs, info = _dyn_run((m, k, n, rp, ci, vals, "bf16", out_dt, B), max_ctas=ctas)
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode("bf16"), B)
    for C in outs:
        assert_parity(C, C_ref, S_ref, f"wcsr dynamic ctas={ctas} N={n}")
    assert np.array_equal(outs[0], outs[1])


def test_wcsr_irregular_dynamic_full_size_sampled():
    """The irregular workload at full size under the dynamic schedule
    (about 1200 chunks of about 62 work items), sampled in every window and
    128-column strip."""
    import sparse_dense_matrix_bcsr_gb300 as S
    w = W.wcsr_irregular()
    outs, info = run_library("wcsr", w.m, w.k, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.B(),
                             keep_device=True, schedule=S.SPMM_SCHEDULE_DYNAMIC)
    import torch
    C = outs[0]
    assert not torch.isnan(C).any().item(), "C not fully written"
    rows, cols = stratified_positions(w.m, w.n, 16, 20000, 5)
    sampled_parity(w, C, rows, cols)


def test_dynamic_schedule_rejected_where_not_built():
    import sparse_dense_matrix_bcsr_gb300 as S
    rng = np.random.default_rng(5)
    rp, ci, vals = W.random_csr(rng, 128, 128, 0.05, "bf16")
    for create, a, b in ((S.spmm_bcsr_create, 64, 64), (S.spmm_wcsr_create, 64, 8)):
        h = create(128, 128, rp, ci, vals, "bf16", "f32", a, b)
        try:
            with pytest.raises(S.SpmmError) as e:
                S.spmm_set_schedule(h, S.SPMM_SCHEDULE_DYNAMIC)
            assert e.value.status == S.SPMM_ERR_UNSUPPORTED
        finally:
            S.spmm_destroy(h)
