"""BCSR product in the layout of a linear layer, Y = X * A^T (spmm_run_linear),
against the oracle: Y is C^T for C = A * B with B = X^T, compared element by
element at small sizes (ragged N, partial block rows and columns, empty block
rows, both input and output types) and at the gate-projection size of the
BCSR weight-like workload (18944 x 3584, 90 % zero blocks, 64K rows of X) on a
sample in every (block row, 256-row tile of X) cell plus whole 256-row bands
of Y."""
import numpy as np
import pytest

import oracle
import spmm_workloads as W
from spmm_testlib import assert_parity, ensure_library, ocode, to_device_bits, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()
    import sparse_dense_matrix_bcsr_gb300 as S
    return S


def run_linear(S, m, k, rp, ci, vals, dt, out_dt, X_bits, runs=1, keep_device=False):
    import torch
    h = S.spmm_bcsr_create(m, k, rp, ci, vals, dt, out_dt)
    try:
        n = X_bits.shape[0]
        dX = to_device_bits(X_bits, dt)
        outs = []
        for _ in range(runs):
            Y = torch.full((n, m), float("nan"), dtype=torch_dtype(out_dt), device="cuda")
            S.spmm_run_linear(h, dX.data_ptr(), Y.data_ptr(), n, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert S.spmm_check(h, torch.cuda.current_stream().cuda_stream) == S.SPMM_OK
            outs.append(Y if keep_device else Y.double().cpu().numpy())
        return outs
    finally:
        S.spmm_destroy(h)


@pytest.mark.parametrize("m,k,n,keep,dt,out_dt", [
    (256, 192, 300, 0.5, "bf16", "bf16"),    # two tiles of X rows, the second ragged
    (640, 512, 1000, 0.3, "bf16", "f32"),
    (200, 200, 257, 0.6, "f16", "f32"),      # partial last block row and column
    (128, 384, 1, 0.5, "bf16", "bf16"),      # a single row of X
    (1024, 256, 2056, 1.0, "f16", "bf16"),   # dense blocks, several tile groups
])
def test_linear_parity_small(S, m, k, n, keep, dt, out_dt):
    rng = np.random.default_rng(m + n)
    rp, ci = W.block_pattern(rng, m, k, 64, 64, keep=keep)
    vals = W.draw_values(rng, len(ci), "u1", dt)
    X = W.dense_bits(rng, (n, k), "u1", dt)
    outs = run_linear(S, m, k, rp, ci, vals, dt, out_dt, X, runs=2)
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode(dt), np.ascontiguousarray(X.T))
    for Y in outs:
        assert_parity(Y.T, C_ref, S_ref, f"linear {m}x{k} N={n}")
    assert np.array_equal(outs[0], outs[1])


def test_linear_empty_block_rows(S):
    rng = np.random.default_rng(7)
    m, k, n = 448, 384, 520
    rp, ci, vals = W.random_csr(rng, m, k, 0.01, "bf16")
    keep = np.ones(len(ci), bool)
    keep[rp[64]:rp[192]] = False
    rows = np.repeat(np.arange(m), np.diff(rp))[keep]
    rp2 = np.zeros(m + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=m), out=rp2[1:])
    X = W.dense_bits(rng, (n, k), "n1", "bf16")
    Y = run_linear(S, m, k, rp2, ci[keep], vals[keep], "bf16", "f32", X)[0]
    C_ref, S_ref = oracle.spmm_csr(m, k, rp2, ci[keep], vals[keep], ocode("bf16"), np.ascontiguousarray(X.T))
    assert_parity(Y.T, C_ref, S_ref, "linear with empty block rows")
    assert np.array_equal(Y[:, 64:192], np.zeros((n, 128)))


def test_linear_rejects_unsupported_shapes(S):
    import torch
    rng = np.random.default_rng(3)
    rp, ci, vals = W.random_csr(rng, 64, 60, 0.1, "bf16")   # k = 60: rows of X not 16-byte multiples
    h = S.spmm_bcsr_create(64, 60, rp, ci, vals, "bf16", "bf16")
    X = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    try:
        with pytest.raises(S.SpmmError) as e:
            S.spmm_run_linear(h, X.data_ptr(), Y.data_ptr(), 8)
        assert e.value.status == S.SPMM_ERR_UNSUPPORTED
    finally:
        S.spmm_destroy(h)
    rp, ci, vals = W.random_csr(rng, 64, 64, 0.1, "bf16")
    h = S.spmm_wcsr_create(64, 64, rp, ci, vals, "bf16", "bf16")
    try:
        with pytest.raises(S.SpmmError) as e:
            S.spmm_run_linear(h, X.data_ptr(), Y.data_ptr(), 8)
        assert e.value.status == S.SPMM_ERR_UNSUPPORTED
    finally:
        S.spmm_destroy(h)


def test_linear_gate_projection_full_size(S):
    import torch
    w = W.bcsr_weight()
    X = np.ascontiguousarray(w.B().T)  # 65536 tokens x 3584 features
    Y = run_linear(S, w.m, w.k, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, X, keep_device=True)[0]
    assert not torch.isnan(Y).any().item(), "Y not fully written"
    rng = np.random.default_rng(0)
    nbr, ntn = -(-w.m // 64), -(-w.n // 256)
    g = np.repeat(np.arange(nbr), ntn)
    t = np.tile(np.arange(ntn), nbr)
    ms = g * 64 + rng.integers(0, 64, len(g))
    ns = t * 256 + rng.integers(0, 256, len(t))
    ms = np.minimum(ms, w.m - 1)
    ns = np.minimum(ns, w.n - 1)
    got = Y[torch.from_numpy(ns).cuda(), torch.from_numpy(ms).cuda()].double().cpu().numpy()
    ref, Sabs = oracle.spmm_csr_sample(w.m, w.k, w.row_ptr, w.col_idx, w.vals, ocode(w.dtype), w.B(), ms, ns)
    assert_parity(got, ref, Sabs, "gate projection sampled")
    B = w.B()
    for n0 in (256 * 100, w.n - 256):
        band = np.ascontiguousarray(B[:, n0:n0 + 256])
        C_ref, S_ref = oracle.spmm_csr(w.m, w.k, w.row_ptr, w.col_idx, w.vals, ocode(w.dtype), band)
        assert_parity(Y[n0:n0 + 256].double().cpu().numpy().T, C_ref, S_ref, f"gate projection rows {n0}..")
