"""Row reordering of A before the WCSR format is built (host preprocessing).

"AsyncSparse", Section IV-A, applies reverse Cuthill-McKee (RCM) to every
matrix before measuring: rows whose columns overlap end up next to each other,
so the fixed-height row windows of WCSR (Section II-C) hold fewer distinct
columns, store fewer padding zeros and gather fewer rows of B.

This module runs on the host, outside the product's hot path, and never
touches the GPU:

    perm = rcm_row_order(m, k, row_ptr, col_idx)      # new row i = old row perm[i]
    rp2, ci2, v2 = permute_rows(row_ptr, col_idx, vals, perm)
    h = spmm_wcsr_create(m, k, rp2, ci2, v2, ...)       # C2 = (P A) B
    # row i of C2 is row perm[i] of C = A B

The ordering is SciPy's reverse_cuthill_mckee on the symmetrised pattern
A + A^T of a square A (the reading of the pages, which reorder square
SuiteSparse matrices), and on the row-overlap graph A A^T for a rectangular
A.  Only rows move: permuting the columns as well would relabel each window's
column set without changing its size.
"""
from __future__ import annotations

import numpy as np


def rcm_row_order(m: int, k: int, row_ptr, col_idx) -> np.ndarray:
    """Reverse Cuthill-McKee order of the rows of A (int64 permutation of
    range(m)); identity for an empty matrix."""
    import scipy.sparse as sp
    from scipy.sparse.csgraph import reverse_cuthill_mckee

    row_ptr = np.asarray(row_ptr, np.int64)
    col_idx = np.asarray(col_idx, np.int32)
    nnz = int(row_ptr[m]) if m else 0
    if m == 0 or nnz == 0:
        return np.arange(m, dtype=np.int64)
    data = np.ones(nnz, np.int8)
    a = sp.csr_matrix((data, col_idx[:nnz], row_ptr), shape=(m, k))
    if m == k:
        g = (a + a.T).tocsr()
    else:
        g = (a @ a.T).tocsr()
    g.sort_indices()
    return np.asarray(reverse_cuthill_mckee(g, symmetric_mode=True), np.int64)


def permute_rows(row_ptr, col_idx, vals, perm):
    """CSR of P A: row i of the result is row perm[i] of A (columns and values
    of each row unchanged).  Returns (row_ptr, col_idx, vals)."""
    row_ptr = np.asarray(row_ptr, np.int64)
    col_idx = np.asarray(col_idx)
    vals = np.asarray(vals)
    perm = np.asarray(perm, np.int64)
    m = len(row_ptr) - 1
    if len(perm) != m or (m and not np.array_equal(np.sort(perm), np.arange(m))):
        raise ValueError("perm must be a permutation of range(m)")
    lens = np.diff(row_ptr)[perm]
    new_ptr = np.zeros(m + 1, np.int64)
    np.cumsum(lens, out=new_ptr[1:])
    starts = row_ptr[perm]
    # source index of every entry of the result, row after row
    src = np.repeat(starts - new_ptr[:-1], lens) + np.arange(new_ptr[-1], dtype=np.int64)
    return new_ptr, col_idx[src], vals[src]


def window_columns(m: int, row_ptr, col_idx, window_h: int = 16) -> int:
    """Distinct columns summed over the row windows of height window_h (the
    WCSR column count before padding): the quantity RCM is meant to lower."""
    row_ptr = np.asarray(row_ptr, np.int64)
    col_idx = np.asarray(col_idx, np.int64)
    rows = np.repeat(np.arange(m, dtype=np.int64), np.diff(row_ptr))
    key = (rows // window_h) * (int(col_idx.max()) + 1 if len(col_idx) else 1) + col_idx
    return int(len(np.unique(key)))
