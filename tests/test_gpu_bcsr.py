"""BCSR kernel parity with the oracle on the GPU (through the C ABI).

Small cases span several 64-row block rows and 128/256-column tiles with
ragged tails and are compared element by element; the full-size benchmark
workloads are compared on seeded samples of outputs that the oracle computes
one by one, and checked for full coverage (no NaN left in a NaN-filled C)."""
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


def full_check(m, k, n, rp, ci, vals, dt, out_dt, B, runs=1):
    outs, info = run_library("bcsr", m, k, rp, ci, vals, dt, out_dt, B, runs=runs)
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode(dt), B)
    for C in outs:
        assert_parity(C, C_ref, S_ref, f"bcsr {m}x{k} N={n}")
    return outs, info


@pytest.mark.parametrize("m,k,n,keep,dt,out_dt", [
    (512, 512, 128, 0.5, "f16", "f32"),     # the BCSR tiny workload's shape
    (300, 200, 72, 0.6, "bf16", "f32"),     # ragged M, K, N < 128
    (640, 448, 264, 0.4, "bf16", "f32"),    # N spans two 256-wide tiles + tail
    (256, 1024, 8, 0.3, "bf16", "f32"),     # N = 8
    (300, 200, 40, 0.6, "bf16", "f32"),     # ragged M, K and N
    (20000, 448, 64, 0.5, "f16", "f32"),    # several tiles per CTA (the stage ring wraps)
    (130, 130, 24, 0.5, "bf16", "bf16"),    # N < 64 with bf16 C
    (192, 320, 256, 1.0, "f16", "bf16"),    # dense blocks everywhere, bf16 C
    (130, 130, 136, 0.5, "bf16", "bf16"),   # partial last block row / column
])
def test_bcsr_parity_small(m, k, n, keep, dt, out_dt):
    rng = np.random.default_rng(m * 31 + n)
    rp, ci = W.block_pattern(rng, m, k, 64, 64, keep=keep)
    vals = W.draw_values(rng, len(ci), "u1", dt)
    B = W.dense_bits(rng, (k, n), "u1", dt)
    full_check(m, k, n, rp, ci, vals, dt, out_dt, B)


@pytest.mark.parametrize("m,k,n,keep,dt,out_dt", [
    (19460, 256, 264, 0.5, "bf16", "bf16"),   # >= 2 tiles per SM: two CTAs per SM, bf16 C, ragged M and N
    (9730, 192, 520, 0.7, "f16", "f32"),      # same path with fp32 C (32-column epilogue parts), 3 column tiles
])
def test_bcsr_parity_two_ctas_per_sm(m, k, n, keep, dt, out_dt):
    """Enough 256-column tiles for the configuration with two CTAs per SM
    (one accumulator each); compared element by element."""
    rng = np.random.default_rng(m + n)
    rp, ci = W.block_pattern(rng, m, k, 64, 64, keep=keep)
    vals = W.draw_values(rng, len(ci), "u1", dt)
    B = W.dense_bits(rng, (k, n), "u1", dt)
    full_check(m, k, n, rp, ci, vals, dt, out_dt, B, runs=2)


@pytest.mark.parametrize("m,k,n,keep,ctas,out_dt", [
    (640, 2048, 264, 0.5, None, "f32"),   # default split grid: 4 stages per CTA, tiles cut into several segments
    (640, 2048, 264, 0.5, 7, "bf16"),     # few CTAs: shares span several tiles and column tiles, bf16 C
    (448, 4096, 128, 0.4, 5, "f32"),      # 128-column tiles (two CTAs per SM, three stages)
    (300, 1024, 72, 0.3, 3, "bf16"),      # ragged M, N < 128
    (64, 4096, 256, 1.0, None, "f32"),    # one block row of 64 blocks: CTA shares inside a single tile
    (200, 640, 520, 0.6, 11, "f32"),      # three 256-column tiles in one group, ragged last tile
])
def test_bcsr_split_schedule(m, k, n, keep, ctas, out_dt):
    """The split schedule (forced here; the automatic choice takes it for few,
    long tiles): equal stage shares per CTA, cut tiles finished by the
    partial-sum pass in CTA order.  Compared element by element and bitwise
    reproducible; the tile schedule on the same input too."""
    rng = np.random.default_rng(m * 7 + n + (ctas or 0))
    rp, ci = W.block_pattern(rng, m, k, 64, 64, keep=keep)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    B = W.dense_bits(rng, (k, n), "u1", "bf16")
    outs, _ = run_library("bcsr", m, k, rp, ci, vals, "bf16", out_dt, B, max_ctas=ctas, runs=2, schedule=2)
    C_ref, S_ref = oracle.spmm_csr(m, k, rp, ci, vals, ocode("bf16"), B)
    for C in outs:
        assert_parity(C, C_ref, S_ref, f"bcsr split {m}x{k} N={n} ctas={ctas}")
    assert np.array_equal(outs[0], outs[1])
    tiles, _ = run_library("bcsr", m, k, rp, ci, vals, "bf16", out_dt, B, max_ctas=ctas, schedule=1)
    assert_parity(tiles[0], C_ref, S_ref, f"bcsr tiles {m}x{k} N={n} ctas={ctas}")


def test_bcsr_many_block_rows_narrow_tiles():
    """Enough block rows for the default (whole-tile) schedule at N <= 128:
    128-column tiles, one CTA per SM, six stages."""
    rng = np.random.default_rng(31)
    m, k, n = 19460, 192, 120
    rp, ci = W.block_pattern(rng, m, k, 64, 64, keep=0.5)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    B = W.dense_bits(rng, (k, n), "u1", "bf16")
    full_check(m, k, n, rp, ci, vals, "bf16", "f32", B, runs=2)


def test_bcsr_tiny_workload():
    w = W.bcsr_tiny()
    outs, info = full_check(w.m, w.k, w.n, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.B(), runs=2)
    assert np.array_equal(outs[0], outs[1])  # deterministic
    assert info["padding"] == 0  # every block is fully populated


def test_bcsr_scattered_entries_and_empty_block_rows():
    """Sparse entries inside blocks (padding zeros stored) and block rows with no block."""
    rng = np.random.default_rng(5)
    m, k, n = 448, 384, 200
    rp, ci, vals = W.random_csr(rng, m, k, 0.01, "bf16")
    # empty out rows 64..191 (two whole block rows)
    keep = np.ones(len(ci), bool)
    keep[rp[64]:rp[192]] = False
    rows = np.repeat(np.arange(m), np.diff(rp))[keep]
    rp2 = np.zeros(m + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=m), out=rp2[1:])
    full_check(m, k, n, rp2, ci[keep], vals[keep], "bf16", "f32", W.dense_bits(rng, (k, n), "n1", "bf16"))


def test_bcsr_identity_exact():
    m = 320
    n = 136
    rp = np.arange(m + 1, dtype=np.int64)
    ci = np.arange(m, dtype=np.int32)
    one = W.f32_to_bf16_bits(np.ones(m, np.float32))
    rng = np.random.default_rng(3)
    B = W.dense_bits(rng, (m, n), "n1", "bf16")
    outs, _ = run_library("bcsr", m, m, rp, ci, one, "bf16", "f32", B)
    assert np.array_equal(outs[0], W.bits_to_f32(B, "bf16").astype(np.float64))


def test_bcsr_one_nonzero_per_row_exact():
    """Products of two 16-bit floats are exact in fp32: C = a_i * B[c_i]."""
    rng = np.random.default_rng(4)
    m, k, n = 200, 500, 64
    rp = np.arange(m + 1, dtype=np.int64)
    ci = np.sort(rng.integers(0, k, m)).astype(np.int32)
    vals = W.draw_values(rng, m, "u1", "f16")
    B = W.dense_bits(rng, (k, n), "u1", "f16")
    outs, _ = run_library("bcsr", m, k, rp, ci, vals, "f16", "f32", B)
    ref = vals.view(np.float16).astype(np.float64)[:, None] * B.view(np.float16).astype(np.float64)[ci]
    assert np.array_equal(outs[0], ref)


def test_bcsr_all_zero_matrix_writes_zeros():
    m, k, n = 130, 70, 24
    rp = np.zeros(m + 1, np.int64)
    B = W.dense_bits(np.random.default_rng(1), (k, n), "u1", "bf16")
    outs, _ = run_library("bcsr", m, k, rp, np.zeros(0, np.int32), np.zeros(0, np.uint16), "bf16", "f32", B)
    assert np.array_equal(outs[0], np.zeros((m, n)))


def sampled_check(w, nsamp=6000, seed=0):
    """Full-size workload: C fully written (no NaN left), then one sampled
    output in every (block row, 128-column strip) cell plus nsamp uniform
    ones compared with the oracle."""
    import torch
    outs, info = run_library("bcsr", w.m, w.k, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.B(),
                             keep_device=True)
    C = outs[0]
    assert not torch.isnan(C).any().item(), "C not fully written"
    rows, cols = stratified_positions(w.m, w.n, 64, nsamp, seed)
    sampled_parity(w, C, rows, cols)
    return info, C


@pytest.mark.parametrize("sp", W.BCSR_SWEEP_SPARSITY)
@pytest.mark.parametrize("n", W.SWEEP_N)
def test_bcsr_sweep_full_size_sampled(sp, n):
    sampled_check(W.bcsr_sweep(sp, n))


def test_bcsr_weight_like_full_size():
    """bcsr_weight at its full size (N = 65536, C bf16): a sample in every
    (block row, 128-column strip) cell, and two whole 256-column bands of C
    (an interior one and the last one) compared element by element."""
    w = W.bcsr_weight()
    info, C = sampled_check(w, nsamp=20000)
    assert info["n_units"] == 1658
    B = w.B()
    for n0 in (256 * 97, w.n - 256):
        band = np.ascontiguousarray(B[:, n0:n0 + 256])
        ref, S = oracle.spmm_csr(w.m, w.k, w.row_ptr, w.col_idx, w.vals, ocode(w.dtype), band)
        got = C[:, n0:n0 + 256].double().cpu().numpy()
        assert_parity(got, ref, S, f"{w.name} columns {n0}..{n0 + 255}")
