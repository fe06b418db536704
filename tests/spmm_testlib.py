"""Shared helpers of the test suite: building the library, moving seeded
inputs to the GPU, running the library through its C ABI and comparing with
the oracle."""
import os

import numpy as np

import oracle
import spmm_workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def ensure_library():
    from sparse_dense_matrix_bcsr_gb300 import build as B
    return B.build()


def ocode(dtype):
    return oracle.BF16 if dtype == "bf16" else oracle.F16


def torch_dtype(name):
    import torch
    return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[name]


def to_device_bits(bits, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch_dtype(dtype))


def run_library(fmt, m, k, rp, ci, vals, dtype, out_dtype, B_bits, b_row=None, b_col=None,
                max_ctas=None, runs=1, keep_device=False, schedule=None):
    """Create a handle, run `runs` times into NaN-filled C, check the device
    status; returns (list of C results as float64 numpy or torch, info)."""
    import torch
    import sparse_dense_matrix_bcsr_gb300 as S
    if fmt == "bcsr":
        h = S.spmm_bcsr_create(m, k, rp, ci, vals, dtype, out_dtype, b_row or 64, b_col or 64)
    else:
        h = S.spmm_wcsr_create(m, k, rp, ci, vals, dtype, out_dtype, b_row or 16, b_col or 16)
    try:
        if max_ctas is not None:
            S.spmm_set_max_ctas(h, max_ctas)
        if schedule is not None:
            S.spmm_set_schedule(h, schedule)
        info = S.spmm_format_info(h)
        N = B_bits.shape[1]
        dB = to_device_bits(B_bits, dtype)
        outs = []
        for _ in range(runs):
            C = torch.full((m, N), float("nan"), dtype=torch_dtype(out_dtype), device="cuda")
            S.run_torch(h, dB, C)
            torch.cuda.synchronize()
            st = S.spmm_check(h, torch.cuda.current_stream().cuda_stream)
            assert st == S.SPMM_OK, S._status_name(st)
            outs.append(C if keep_device else C.double().cpu().numpy())
        return outs, info
    finally:
        S.spmm_destroy(h)


def assert_parity(C_gpu, C_ref, S_ref, what=""):
    ok, worst = oracle.within_tolerance(C_gpu, C_ref, S_ref)
    assert ok, f"{what}: |err| exceeds 4*2^-8*S + 1e-6 (worst err/bound = {worst:.3g})"
    return worst


def stratified_positions(m, n, group_rows, nsamp_random=0, seed=0, strata_cols=128):
    """Sample positions of C: one random (row, column) inside every
    (row group, column stratum) cell -- a BCSR block row or WCSR window by a
    strip of `strata_cols` columns, finer than either kernel's column tile --
    plus `nsamp_random` uniform positions.  Every tile the kernels write is
    therefore sampled at least once."""
    rng = np.random.default_rng(seed)
    ng = -(-m // group_rows)
    nc = -(-n // strata_cols)
    g = np.repeat(np.arange(ng, dtype=np.int64), nc)
    c = np.tile(np.arange(nc, dtype=np.int64), ng)
    r0 = g * group_rows
    rows = r0 + (rng.random(len(g)) * np.minimum(group_rows, m - r0)).astype(np.int64)
    c0 = c * strata_cols
    cols = c0 + (rng.random(len(c)) * np.minimum(strata_cols, n - c0)).astype(np.int64)
    if nsamp_random:
        rows = np.concatenate([rows, rng.integers(0, m, nsamp_random)])
        cols = np.concatenate([cols, rng.integers(0, n, nsamp_random)])
    return rows, cols


def sampled_parity(w, C_dev, rows, cols):
    """Compare C_dev (a torch tensor on the GPU) with the oracle at (rows, cols)."""
    import torch
    Cs = C_dev[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    ref, S = oracle.spmm_csr_sample(w.m, w.k, w.row_ptr, w.col_idx, w.vals, ocode(w.dtype), w.B(), rows, cols)
    return assert_parity(Cs, ref, S, f"{w.name} ({len(rows)} sampled outputs)")
