"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one oracle function to something the paper or mathematics
fixes: the Fig. 2 index arrays of "AsyncSparse" (Section II-C), brute-force
enumeration from a dense copy, a dense fp64 matrix product computed by numpy,
closed forms (identity, one nonzero per row), and the storage invariant
stored = nnz + padding.  The last tests plant mistakes in oracle outputs and
check that the pins reject them.
"""
import json
import os

import numpy as np
import pytest

import oracle
import spmm_workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fig2_formats.json")


def _dtype_code(dt):
    return oracle.BF16 if dt == "bf16" else oracle.F16


def densify(m, k, rp, ci, vals, dtype):
    """Dense float64 copy of a CSR (bits decoded by numpy, not by the oracle)."""
    A = np.zeros((m, k), np.float64)
    mask = np.zeros((m, k), bool)
    for i in range(m):
        cols = ci[rp[i]:rp[i + 1]]
        A[i, cols] = W.bits_to_f32(vals[rp[i]:rp[i + 1]], dtype).astype(np.float64)
        mask[i, cols] = True
    return A, mask


def dense_bits_of(m, k, rp, ci, vals):
    D = np.zeros((m, k), np.uint16)
    for i in range(m):
        D[i, ci[rp[i]:rp[i + 1]]] = vals[rp[i]:rp[i + 1]]
    return D


def fig2():
    with open(GOLDEN) as f:
        g = json.load(f)
    m, k = g["m"], g["k"]
    rp = np.zeros(m + 1, np.int64)
    cols = []
    for i, r in enumerate(g["rows"]):
        rp[i + 1] = rp[i] + len(r)
        cols += r
    ci = np.array(cols, np.int32)
    vals = W.f32_to_f16_bits(np.arange(1, len(ci) + 1, dtype=np.float32))
    return g, m, k, rp, ci, vals


# ------------------------------------------------------------ Fig. 2 arrays
def test_fig2_bcsr_index_arrays():
    g, m, k, rp, ci, vals = fig2()
    brp, bci, blocks = oracle.bcsr_build(m, k, rp, ci, vals, g["b_row"], g["b_col"])
    assert brp.tolist() == g["expected"]["block_row_ptr"]
    assert bci.tolist() == g["expected"]["block_col_idx"]
    assert blocks.shape == (5, 4, 4)


def test_fig2_wcsr_index_arrays():
    g, m, k, rp, ci, vals = fig2()
    wrp, wci, values = oracle.wcsr_build(m, k, rp, ci, vals, g["b_row"], g["b_col"])
    assert wrp.tolist() == g["expected"]["window_row_ptr"]
    assert wci.tolist() == g["expected"]["window_col_idx"]
    assert values.shape == (4, 12)
    # 15 values stored, 4*12 - 15 padding slots hold +0.
    assert int((values != 0).sum()) == 15


# ------------------------------------------------------------ half decoding
def test_f16_decoding_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(b, oracle.F16) for b in bits[::7]])
    r = ref[::7]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], r[~nan])
    # special patterns
    assert oracle.half_to_double(0x3C00, oracle.F16) == 1.0
    assert oracle.half_to_double(0xC000, oracle.F16) == -2.0
    assert oracle.half_to_double(0x0001, oracle.F16) == 2.0 ** -24
    assert oracle.half_to_double(0x7BFF, oracle.F16) == 65504.0


def test_bf16_decoding_is_upper_half_of_f32():
    for b in (0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F, 0x8000):
        ref = float(np.array([b << 16], np.uint32).view(np.float32)[0])
        assert oracle.half_to_double(b, oracle.BF16) == ref
    assert oracle.half_to_double(0x3F80, oracle.BF16) == 1.0


# ------------------------------------------------------------ CSR validity
def test_csr_check():
    ok = oracle.csr_check(2, 4, [0, 2, 3], [0, 3, 1])
    assert ok == 0
    assert oracle.csr_check(2, 4, [1, 2, 3], [0, 3, 1]) == 1          # row_ptr[0] != 0
    assert oracle.csr_check(2, 4, [0, 2, 1], [0, 3, 1]) == 1          # decreasing
    assert oracle.csr_check(2, 4, [0, 2, 3], [0, 4, 1]) == 2          # column == k
    assert oracle.csr_check(2, 4, [0, 2, 3], [0, -1, 1]) == 2         # negative column
    assert oracle.csr_check(2, 4, [0, 2, 3], [3, 0, 1]) == 3          # unsorted
    assert oracle.csr_check(2, 4, [0, 2, 3], [2, 2, 1]) == 3          # duplicate
    assert oracle.csr_check(0, 4, [0], []) == 0                       # empty matrix


# ------------------------------------------------------------ brute force
CASES = [
    # m, k, density, b_row, b_col, dtype
    (37, 53, 0.10, 8, 8, "bf16"),
    (64, 64, 0.02, 16, 16, "f16"),
    (130, 70, 0.05, 64, 64, "bf16"),
    (5, 200, 0.30, 4, 32, "f16"),
    (100, 100, 0.0, 16, 16, "bf16"),   # empty matrix
    (33, 17, 1.0, 16, 16, "bf16"),     # full matrix, ragged edges
    (150, 90, 0.05, 64, 8, "bf16"),    # the pages' WCSR geometry: 64-row windows, padding 8
]


@pytest.mark.parametrize("m,k,d,br,bc,dt", CASES)
def test_bcsr_brute_force(m, k, d, br, bc, dt):
    rng = np.random.default_rng(11 + m + k)
    rp, ci, vals = W.random_csr(rng, m, k, d, dt)
    D = dense_bits_of(m, k, rp, ci, vals)
    _, mask = densify(m, k, rp, ci, vals, dt)
    brp, bci, blocks = oracle.bcsr_build(m, k, rp, ci, vals, br, bc)
    nbr, nbc = -(-m // br), -(-k // bc)
    exp_ptr = [0]
    exp_idx = []
    exp_blocks = []
    for R in range(nbr):
        for C in range(nbc):
            sub = mask[R * br:(R + 1) * br, C * bc:(C + 1) * bc]
            if sub.any():
                exp_idx.append(C)
                blk = np.zeros((br, bc), np.uint16)
                s = D[R * br:(R + 1) * br, C * bc:(C + 1) * bc]
                blk[:s.shape[0], :s.shape[1]] = s
                exp_blocks.append(blk)
        exp_ptr.append(len(exp_idx))
    assert brp.tolist() == exp_ptr
    assert bci.tolist() == exp_idx
    if exp_blocks:
        assert np.array_equal(blocks, np.stack(exp_blocks))
    # stored = nnz + padding, and every stored nonzero is a CSR entry
    nnz = len(ci)
    stored = blocks.size
    padding = int((blocks & 0x7FFF == 0).sum())
    assert stored == nnz + padding
    if stored:
        fill = nnz / stored
        assert 0 < fill <= 1


@pytest.mark.parametrize("m,k,d,h,pad,dt", CASES)
def test_wcsr_brute_force(m, k, d, h, pad, dt):
    rng = np.random.default_rng(23 + m + k)
    rp, ci, vals = W.random_csr(rng, m, k, d, dt)
    D = dense_bits_of(m, k, rp, ci, vals)
    _, mask = densify(m, k, rp, ci, vals, dt)
    wrp, wci, values = oracle.wcsr_build(m, k, rp, ci, vals, h, pad)
    nw = -(-m // h)
    exp_ptr = [0]
    exp_idx = []
    for w in range(nw):
        cols = [c for c in range(k) if mask[w * h:(w + 1) * h, c].any()]
        P = -(-len(cols) // pad) * pad
        exp_idx += cols + [-1] * (P - len(cols))
        exp_ptr.append(len(exp_idx))
    assert wrp.tolist() == exp_ptr
    assert wci.tolist() == exp_idx
    Ptot = len(exp_idx)
    assert values.shape == (h, Ptot)
    for w in range(nw):
        for p in range(exp_ptr[w], exp_ptr[w + 1]):
            c = exp_idx[p]
            for r in range(h):
                i = w * h + r
                want = D[i, c] if (c >= 0 and i < m) else 0
                assert values[r, p] == want
    nnz = len(ci)
    padding = int((values & 0x7FFF == 0).sum())
    assert values.size == nnz + padding


# ------------------------------------------------------------ SpMM
@pytest.mark.parametrize("m,k,n,d,dt", [(40, 70, 24, 0.1, "bf16"), (64, 64, 8, 0.3, "f16"),
                                         (1, 300, 5, 0.5, "bf16"), (90, 3, 17, 0.6, "f16"),
                                         (20, 20, 4, 0.0, "bf16")])
def test_spmm_matches_dense_matmul(m, k, n, d, dt):
    rng = np.random.default_rng(7 * m + n)
    rp, ci, vals = W.random_csr(rng, m, k, d, dt)
    B = W.dense_bits(rng, (k, n), "n1", dt)
    A, _ = densify(m, k, rp, ci, vals, dt)
    Bf = W.bits_to_f32(B, dt).astype(np.float64)
    C, S = oracle.spmm_csr(m, k, rp, ci, vals, _dtype_code(dt), B)
    ref = A @ Bf
    refS = np.abs(A) @ np.abs(Bf)
    assert np.all(np.abs(C - ref) <= 1e-12 * refS + 1e-300)
    assert np.allclose(S, refS, rtol=1e-12, atol=0)


def test_spmm_identity_is_exact():
    n = 33
    m = 50
    rp = np.arange(m + 1, dtype=np.int64)
    ci = np.arange(m, dtype=np.int32)
    one = W.f32_to_bf16_bits(np.ones(m, np.float32))
    rng = np.random.default_rng(5)
    B = W.dense_bits(rng, (m, n), "n1", "bf16")
    C, S = oracle.spmm_csr(m, m, rp, ci, one, oracle.BF16, B)
    Bf = W.bits_to_f32(B, "bf16").astype(np.float64)
    assert np.array_equal(C, Bf)
    assert np.array_equal(S, np.abs(Bf))


def test_spmm_one_nonzero_per_row_is_exact():
    rng = np.random.default_rng(6)
    m, k, n = 70, 40, 19
    rp = np.arange(m + 1, dtype=np.int64)
    ci = rng.integers(0, k, m).astype(np.int32)
    vals = W.draw_values(rng, m, "u1", "f16")
    B = W.dense_bits(rng, (k, n), "u1", "f16")
    C, _ = oracle.spmm_csr(m, k, rp, ci, vals, oracle.F16, B)
    a = vals.view(np.float16).astype(np.float64)
    Bf = B.view(np.float16).astype(np.float64)
    assert np.array_equal(C, a[:, None] * Bf[ci])


def test_sample_matches_full():
    rng = np.random.default_rng(8)
    m, k, n = 60, 80, 12
    rp, ci, vals = W.random_csr(rng, m, k, 0.2, "bf16")
    B = W.dense_bits(rng, (k, n), "n1", "bf16")
    C, S = oracle.spmm_csr(m, k, rp, ci, vals, oracle.BF16, B)
    rows = rng.integers(0, m, 200)
    cols = rng.integers(0, n, 200)
    Cs, Ss = oracle.spmm_csr_sample(m, k, rp, ci, vals, oracle.BF16, B, rows, cols)
    assert np.array_equal(Cs, C[rows, cols])
    assert np.array_equal(Ss, S[rows, cols])


@pytest.mark.parametrize("m,k,n,d,br,bc", [(70, 90, 16, 0.1, 16, 16), (128, 128, 8, 0.05, 64, 64),
                                             (33, 65, 9, 0.3, 8, 4)])
def test_format_spmm_matches_csr(m, k, n, d, br, bc):
    rng = np.random.default_rng(m * k)
    rp, ci, vals = W.random_csr(rng, m, k, d, "bf16")
    B = W.dense_bits(rng, (k, n), "n1", "bf16")
    C, S = oracle.spmm_csr(m, k, rp, ci, vals, oracle.BF16, B)
    brp, bci, blocks = oracle.bcsr_build(m, k, rp, ci, vals, br, bc)
    Cb = oracle.spmm_bcsr(m, k, brp, bci, blocks, oracle.BF16, B)
    wrp, wci, values = oracle.wcsr_build(m, k, rp, ci, vals, br, bc)
    Cw = oracle.spmm_wcsr(m, k, wrp, wci, values, oracle.BF16, B)
    assert np.all(np.abs(Cb - C) <= 1e-12 * S)
    assert np.all(np.abs(Cw - C) <= 1e-12 * S)


def test_block_diagonal_bcsr_is_independent_gemms():
    """A block-diagonal A: each block row's product is one dense GEMM."""
    rng = np.random.default_rng(9)
    nb, b, n = 3, 16, 10
    m = nb * b
    blocks = [W.dense_bits(rng, (b, b), "u1", "bf16") for _ in range(nb)]
    rows, cols, vals = [], [], []
    for t, blk in enumerate(blocks):
        for r in range(b):
            for c in range(b):
                rows.append(t * b + r)
                cols.append(t * b + c)
                vals.append(blk[r, c])
    rp = np.zeros(m + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=m), out=rp[1:])
    ci = np.array(cols, np.int32)
    vv = np.array(vals, np.uint16)
    B = W.dense_bits(rng, (m, n), "u1", "bf16")
    brp, bci, bl = oracle.bcsr_build(m, m, rp, ci, vv, b, b)
    assert brp.tolist() == [0, 1, 2, 3] and bci.tolist() == [0, 1, 2]
    C = oracle.spmm_bcsr(m, m, brp, bci, bl, oracle.BF16, B)
    Bf = W.bits_to_f32(B, "bf16").astype(np.float64)
    for t in range(nb):
        Ab = W.bits_to_f32(blocks[t], "bf16").astype(np.float64)
        ref = Ab @ Bf[t * b:(t + 1) * b]
        assert np.allclose(C[t * b:(t + 1) * b], ref, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------ tolerance
def test_tolerance_rule():
    ref = np.array([1.0, -2.0, 0.0])
    S = np.array([1.0, 4.0, 0.0])
    ok, _ = oracle.within_tolerance(ref + np.array([0.015, -0.06, 5e-7]), ref, S)
    assert ok
    ok, _ = oracle.within_tolerance(ref + np.array([0.0, 0.07, 0.0]), ref, S)
    assert not ok
    ok, _ = oracle.within_tolerance(np.array([np.nan, -2.0, 0.0]), ref, S)
    assert not ok


# ------------------------------------------------------------ planted mistakes
def test_pins_reject_planted_mistakes():
    """Plausible oracle bugs -- a dropped term, a transposed operand, a wrong
    sign, an off-by-one column -- all fail the dense-matmul pin."""
    rng = np.random.default_rng(10)
    m = k = 24
    n = 6
    rp, ci, vals = W.random_csr(rng, m, k, 0.25, "bf16")
    B = W.dense_bits(rng, (k, n), "n1", "bf16")
    A, _ = densify(m, k, rp, ci, vals, "bf16")
    Bf = W.bits_to_f32(B, "bf16").astype(np.float64)
    ref = A @ Bf
    refS = np.abs(A) @ np.abs(Bf)

    def passes(C):
        return bool(np.all(np.abs(C - ref) <= 1e-12 * refS + 1e-300))

    C, _ = oracle.spmm_csr(m, k, rp, ci, vals, oracle.BF16, B)
    assert passes(C)
    # dropped last term of each row
    v2 = vals.copy()
    v2[rp[1:][np.diff(rp) > 0] - 1] = 0
    C2, _ = oracle.spmm_csr(m, k, rp, ci, v2, oracle.BF16, B)
    assert not passes(C2)
    # transposed A
    At = A.T.copy()
    assert not passes(At @ Bf)
    # sign flip of one entry
    v3 = vals.copy()
    v3[0] ^= 0x8000
    C3, _ = oracle.spmm_csr(m, k, rp, ci, v3, oracle.BF16, B)
    assert not passes(C3)
    # off-by-one column index
    ci4 = np.minimum(ci + 1, k - 1).astype(np.int32)
    C4, _ = oracle.spmm_csr(m, k, rp, ci4, vals, oracle.BF16, B)
    assert not passes(C4)
