"""Host preprocessing: reverse Cuthill-McKee row order before building WCSR
("AsyncSparse", Section IV-A).  Checked on the CPU: the row permutation of a
CSR against the dense matrix, RCM recovering a banded matrix from a symmetric
relabelling (its window column count drops back), and the product of the
permuted matrix equal to the permuted rows of the original product (oracle)."""
import numpy as np
import pytest

import oracle
import spmm_workloads as W
from sparse_dense_matrix_bcsr_gb300 import reorder as R

pytest.importorskip("scipy")


def dense(m, k, rp, ci, vals):
    d = np.zeros((m, k), np.uint16)
    rows = np.repeat(np.arange(m), np.diff(rp))
    d[rows, ci] = vals
    return d


def test_permute_rows_matches_dense():
    rng = np.random.default_rng(1)
    m, k = 37, 50
    rp, ci, vals = W.random_csr(rng, m, k, 0.2)
    perm = rng.permutation(m)
    rp2, ci2, v2 = R.permute_rows(rp, ci, vals, perm)
    assert np.array_equal(dense(m, k, rp2, ci2, v2), dense(m, k, rp, ci, vals)[perm])
    assert oracle.csr_check(m, k, rp2, ci2) == 0
    with pytest.raises(ValueError):
        R.permute_rows(rp, ci, vals, np.zeros(m, np.int64))


def test_rcm_recovers_a_banded_matrix_from_a_symmetric_relabelling():
    """A banded square matrix whose rows and columns were relabelled by the
    same random permutation: its 16-row windows hold many distinct columns;
    RCM on A + A^T finds a banded order again, and moving only the rows to it
    brings the windows' column count back near the banded one."""
    rng = np.random.default_rng(2)
    m = 2048
    band = 6
    rows, cols = [], []
    for i in range(m):
        c = np.arange(max(0, i - band), min(m, i + band + 1))
        rows.append(np.full(len(c), i))
        cols.append(c)
    rows = np.concatenate(rows)
    cols = np.concatenate(cols)
    banded = R.window_columns(m, *csr_of(m, rows, cols))
    q = rng.permutation(m)          # old label -> new label
    rp_s, ci_s = csr_of(m, q[rows], q[cols])
    vals = W.draw_values(rng, len(ci_s), "u1", "bf16")
    relabelled = R.window_columns(m, rp_s, ci_s)
    perm = R.rcm_row_order(m, m, rp_s, ci_s)
    assert np.array_equal(np.sort(perm), np.arange(m))
    rp_r, ci_r, _ = R.permute_rows(rp_s, ci_s, vals, perm)
    rcm = R.window_columns(m, rp_r, ci_r)
    assert relabelled > 5 * banded
    assert rcm < 1.5 * banded


def csr_of(m, rows, cols):
    order = np.lexsort((cols, rows))
    rp = np.zeros(m + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=m), out=rp[1:])
    return rp, np.asarray(cols)[order].astype(np.int32)


@pytest.mark.parametrize("m,k", [(300, 300), (200, 500)])
def test_product_of_reordered_matrix_is_reordered_product(m, k):
    rng = np.random.default_rng(m + k)
    rp, ci = W.powerlaw_pattern(rng, m, k, 1.5, 1, 60, 20, 0.7)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    B = W.dense_bits(rng, (k, 24), "u1", "bf16")
    perm = R.rcm_row_order(m, k, rp, ci)
    rp2, ci2, v2 = R.permute_rows(rp, ci, vals, perm)
    C, _ = oracle.spmm_csr(m, k, rp, ci, vals, oracle.BF16, B)
    C2, _ = oracle.spmm_csr(m, k, rp2, ci2, v2, oracle.BF16, B)
    assert np.array_equal(C2, C[perm])


def test_empty_matrix_keeps_identity_order():
    rp = np.zeros(9, np.int64)
    assert np.array_equal(R.rcm_row_order(8, 8, rp, np.zeros(0, np.int32)), np.arange(8))
