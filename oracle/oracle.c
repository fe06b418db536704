/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for sparse x dense
 * matrix multiplication C = A * B with A sparse (CSR) and B, C dense, and for
 * the two sparse formats of "AsyncSparse: Accelerating Sparse Matrix-Matrix
 * Multiplication on Asynchronous GPU Architectures" (Liu, Pu, Zhang),
 * Section II-C and Fig. 2: BCSR (Block Compressed Sparse Row) and WCSR
 * (Window Compressed Sparse Row).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load or call this code.  The library's
 * GPU path shares nothing with it: no code, no header, no table.
 *
 * Conventions
 *   - A is m x k in CSR: row_ptr[m+1] (int64), col_idx[nnz] (int32), vals[nnz]
 *     given as the raw bits of a 16-bit float (fp16 or bf16).
 *   - B is k x n row-major, 16-bit bits of the same type; C is m x n row-major.
 *   - All products and sums are taken in double precision (fp64).
 *   - Every explicit CSR entry is a structural nonzero, even if its value is 0.
 *
 * Readings of the paper made here (the paper is silent or garbled on them):
 *   - The number of block rows / windows is ceil(m / b_row), columns of blocks
 *     ceil(k / b_col); a partial last block or window is zero-padded.
 *   - BCSR blocks are kept in ascending block-column order within a block row
 *     (Fig. 2), each block dense row-major b_row x b_col.
 *   - WCSR window column lists are the ascending union of the window's
 *     columns, followed by -1 entries up to a multiple of b_col (Fig. 2).
 *     window_row_ptr counts padded column positions (Fig. 2: [0,4,12]).
 *   - WCSR values are ONE row-major array of shape [b_row][P_total], P_total
 *     being the total padded column count; element (r, p) is
 *     A[b_row*w + r][window_col_idx[p]] for the window w owning position p,
 *     0 where that entry is absent, the column is padding, or the row is past m.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F16 0
#define ORC_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE 754 binary32. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

double orc_half_to_double(uint16_t bits, int dtype) {
    return dtype == ORC_BF16 ? bf16_bits_to_double(bits) : f16_bits_to_double(bits);
}

/* Decoding table for all 65536 bit patterns of one dtype. */
static double *decode_table(int dtype) {
    double *t = (double *)malloc(65536 * sizeof(double));
    if (!t) return NULL;
    for (uint32_t b = 0; b < 65536; ++b) t[b] = orc_half_to_double((uint16_t)b, dtype);
    return t;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/*
 * CSR validity: row_ptr[0] == 0, row_ptr non-decreasing, row_ptr[m] == nnz
 * (not checked here: the caller gives nnz implicitly), every column in
 * [0, k), and columns strictly ascending within each row.
 * Returns 0 if valid, 1 bad row_ptr, 2 column out of range, 3 unsorted or
 * duplicate column.
 */
int orc_csr_check(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx) {
    if (m < 0 || k < 0) return 1;
    if (row_ptr[0] != 0) return 1;
    for (int64_t i = 0; i < m; ++i)
        if (row_ptr[i + 1] < row_ptr[i]) return 1;
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
            if (col_idx[e] < 0 || (int64_t)col_idx[e] >= k) return 2;
            if (e > row_ptr[i] && col_idx[e] <= col_idx[e - 1]) return 3;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ BCSR --
 * BCSR (paper Section II-C, "Block Compressed Sparse Row"; Fig. 2): A is cut
 * into b_row x b_col blocks; a block is stored (dense) iff it holds at least
 * one nonzero.  block_row_ptr[ceil(m/b_row)+1] starts each block row's run
 * of stored blocks, block_col_idx[nnz_blocks] is each stored block's block
 * column, blocks[nnz_blocks * b_row * b_col] their dense values.
 */

/* Mark, for block row R, which block columns hold a nonzero.  occ has
 * ceil(k/b_col) entries and is overwritten. */
static void bcsr_occupancy(int64_t m, int64_t R, int b_row, int b_col, int64_t nbc,
                           const int64_t *row_ptr, const int32_t *col_idx, char *occ) {
    memset(occ, 0, (size_t)nbc);
    int64_t r0 = R * b_row, r1 = r0 + b_row < m ? r0 + b_row : m;
    for (int64_t i = r0; i < r1; ++i)
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) occ[col_idx[e] / b_col] = 1;
}

/* Number of stored blocks. */
int64_t orc_bcsr_nblocks(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                         int b_row, int b_col) {
    int64_t nbr = ceil_div(m, b_row), nbc = ceil_div(k, b_col), total = 0;
    char *occ = (char *)malloc((size_t)(nbc > 0 ? nbc : 1));
    for (int64_t R = 0; R < nbr; ++R) {
        bcsr_occupancy(m, R, b_row, b_col, nbc, row_ptr, col_idx, occ);
        for (int64_t c = 0; c < nbc; ++c) total += occ[c];
    }
    free(occ);
    return total;
}

/* Fill the three BCSR arrays; blocks holds the input's 16-bit bits verbatim
 * and 0 (+0.0) elsewhere.  Arrays are sized by orc_bcsr_nblocks. */
void orc_bcsr_build(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                    const uint16_t *vals, int b_row, int b_col, int64_t *block_row_ptr,
                    int32_t *block_col_idx, uint16_t *blocks) {
    int64_t nbr = ceil_div(m, b_row), nbc = ceil_div(k, b_col);
    int64_t bsz = (int64_t)b_row * b_col;
    char *occ = (char *)malloc((size_t)(nbc > 0 ? nbc : 1));
    int64_t nb = 0;
    block_row_ptr[0] = 0;
    for (int64_t R = 0; R < nbr; ++R) {
        bcsr_occupancy(m, R, b_row, b_col, nbc, row_ptr, col_idx, occ);
        int64_t first = nb;
        for (int64_t c = 0; c < nbc; ++c)
            if (occ[c]) {
                block_col_idx[nb] = (int32_t)c;
                memset(blocks + nb * bsz, 0, (size_t)bsz * sizeof(uint16_t));
                ++nb;
            }
        block_row_ptr[R + 1] = nb;
        /* Place each entry of the block row into its block. */
        int64_t r0 = R * b_row, r1 = r0 + b_row < m ? r0 + b_row : m;
        for (int64_t i = r0; i < r1; ++i)
            for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
                int32_t bc = col_idx[e] / b_col;
                int64_t j = first;
                while (block_col_idx[j] != bc) ++j; /* linear search: it is there */
                blocks[j * bsz + (i - r0) * b_col + (col_idx[e] - (int64_t)bc * b_col)] = vals[e];
            }
    }
    free(occ);
}

/* ------------------------------------------------------------------ WCSR --
 * WCSR (paper Section II-C, "Window Compressed Sparse Row"; Fig. 2): rows are
 * grouped into windows of b_row rows; each window keeps the union of the
 * column indices of its rows, padded with -1 to a multiple of b_col.
 * window_row_ptr[ceil(m/b_row)+1] starts each window's padded column run,
 * window_col_idx[P_total] names the original column of each position (-1 for
 * padding), values holds the packed values (layout: see the file header).
 */

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Sorted distinct columns of window w, written to buf (capacity: the window's
 * nnz); returns their count. */
static int64_t window_union(int64_t m, int64_t w, int h, const int64_t *row_ptr,
                            const int32_t *col_idx, int32_t *buf) {
    int64_t r0 = w * h, r1 = r0 + h < m ? r0 + h : m, n = 0;
    for (int64_t i = r0; i < r1; ++i)
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) buf[n++] = col_idx[e];
    qsort(buf, (size_t)n, sizeof(int32_t), cmp_i32);
    int64_t u = 0;
    for (int64_t j = 0; j < n; ++j)
        if (u == 0 || buf[j] != buf[u - 1]) buf[u++] = buf[j];
    return u;
}

static int64_t window_nnz(int64_t m, int64_t w, int h, const int64_t *row_ptr) {
    int64_t r0 = w * h, r1 = r0 + h < m ? r0 + h : m;
    return row_ptr[r1] - row_ptr[r0];
}

/* Total padded column positions P_total. */
int64_t orc_wcsr_ncols(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                       int h, int pad) {
    (void)k;
    int64_t nw = ceil_div(m, h), total = 0;
    for (int64_t w = 0; w < nw; ++w) {
        int64_t wn = window_nnz(m, w, h, row_ptr);
        int32_t *buf = (int32_t *)malloc((size_t)(wn > 0 ? wn : 1) * sizeof(int32_t));
        int64_t u = window_union(m, w, h, row_ptr, col_idx, buf);
        total += ceil_div(u, pad) * pad;
        free(buf);
    }
    return total;
}

/* Fill the three WCSR arrays; values is [h][P_total] row-major, P_total from
 * orc_wcsr_ncols. */
void orc_wcsr_build(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                    const uint16_t *vals, int h, int pad, int64_t *window_row_ptr,
                    int32_t *window_col_idx, uint16_t *values) {
    int64_t nw = ceil_div(m, h);
    int64_t P = orc_wcsr_ncols(m, k, row_ptr, col_idx, h, pad);
    memset(values, 0, (size_t)(P * h) * sizeof(uint16_t));
    int64_t pos = 0;
    window_row_ptr[0] = 0;
    for (int64_t w = 0; w < nw; ++w) {
        int64_t wn = window_nnz(m, w, h, row_ptr);
        int32_t *buf = (int32_t *)malloc((size_t)(wn > 0 ? wn : 1) * sizeof(int32_t));
        int64_t u = window_union(m, w, h, row_ptr, col_idx, buf);
        int64_t pw = ceil_div(u, pad) * pad;
        for (int64_t j = 0; j < pw; ++j) window_col_idx[pos + j] = j < u ? buf[j] : -1;
        int64_t r0 = w * h, r1 = r0 + h < m ? r0 + h : m;
        for (int64_t i = r0; i < r1; ++i)
            for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
                /* position of this column within the window's union */
                int32_t *hit = (int32_t *)bsearch(&col_idx[e], buf, (size_t)u, sizeof(int32_t), cmp_i32);
                int64_t p = pos + (hit - buf);
                values[(i - r0) * P + p] = vals[e];
            }
        pos += pw;
        window_row_ptr[w + 1] = pos;
        free(buf);
    }
}

/* ------------------------------------------------------------------ SpMM --
 * C = A * B from the CSR itself, by the definition C[i][j] = sum over the
 * stored entries (i, c, a) of a * B[c][j], in fp64; S[i][j] is the same sum
 * of |a * B[c][j]|, used for the error bound of the parity tests.  The
 * paper's problem statement (Section II-C: C = A x B, A m x k sparse).
 * Rows are independent; OpenMP splits them across `threads` threads
 * (threads <= 0: the OpenMP default).
 */
void orc_spmm_csr(int64_t m, int64_t k, int64_t n, const int64_t *row_ptr,
                  const int32_t *col_idx, const uint16_t *vals, int dtype, const uint16_t *B,
                  double *C, double *S, int threads) {
    (void)k;
    double *tab = decode_table(dtype);
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t i = 0; i < m; ++i) {
        double *c = C + i * n;
        double *s = S ? S + i * n : NULL;
        for (int64_t j = 0; j < n; ++j) c[j] = 0.0;
        if (s)
            for (int64_t j = 0; j < n; ++j) s[j] = 0.0;
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
            double a = tab[vals[e]];
            const uint16_t *b = B + (int64_t)col_idx[e] * n;
            for (int64_t j = 0; j < n; ++j) {
                double p = a * tab[b[j]];
                c[j] += p;
                if (s) s[j] += fabs(p);
            }
        }
    }
    free(tab);
}

/* The same sums for a list of output positions (rows[t], cols[t]). */
void orc_spmm_csr_sample(int64_t m, int64_t k, int64_t n, const int64_t *row_ptr,
                         const int32_t *col_idx, const uint16_t *vals, int dtype,
                         const uint16_t *B, int64_t nsamp, const int64_t *rows,
                         const int64_t *cols, double *C, double *S) {
    (void)m;
    (void)k;
    double *tab = decode_table(dtype);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t t = 0; t < nsamp; ++t) {
        int64_t i = rows[t], j = cols[t];
        double c = 0.0, s = 0.0;
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
            double p = tab[vals[e]] * tab[B[(int64_t)col_idx[e] * n + j]];
            c += p;
            s += fabs(p);
        }
        C[t] = c;
        S[t] = s;
    }
    free(tab);
}

/* C = A * B computed from the BCSR arrays: every stored block (dense,
 * zeros included) times its b_col rows of B.  Cross-checks the converter. */
void orc_spmm_bcsr(int64_t m, int64_t k, int64_t n, int b_row, int b_col,
                   const int64_t *block_row_ptr, const int32_t *block_col_idx,
                   const uint16_t *blocks, int dtype, const uint16_t *B, double *C) {
    double *tab = decode_table(dtype);
    int64_t nbr = ceil_div(m, b_row), bsz = (int64_t)b_row * b_col;
    for (int64_t x = 0; x < m * n; ++x) C[x] = 0.0;
    for (int64_t R = 0; R < nbr; ++R)
        for (int64_t j = block_row_ptr[R]; j < block_row_ptr[R + 1]; ++j)
            for (int64_t r = 0; r < b_row; ++r) {
                int64_t i = R * b_row + r;
                if (i >= m) break;
                for (int64_t cc = 0; cc < b_col; ++cc) {
                    int64_t col = (int64_t)block_col_idx[j] * b_col + cc;
                    if (col >= k) break;
                    double a = tab[blocks[j * bsz + r * b_col + cc]];
                    for (int64_t q = 0; q < n; ++q) C[i * n + q] += a * tab[B[col * n + q]];
                }
            }
    free(tab);
}

/* C = A * B computed from the WCSR arrays: every packed position p of window
 * w contributes values[r][p] * B[window_col_idx[p]][:] to row h*w + r;
 * padding positions (-1) contribute nothing.  Cross-checks the converter. */
void orc_spmm_wcsr(int64_t m, int64_t k, int64_t n, int h, const int64_t *window_row_ptr,
                   const int32_t *window_col_idx, const uint16_t *values, int dtype,
                   const uint16_t *B, double *C) {
    (void)k;
    double *tab = decode_table(dtype);
    int64_t nw = ceil_div(m, h), P = window_row_ptr[nw];
    for (int64_t x = 0; x < m * n; ++x) C[x] = 0.0;
    for (int64_t w = 0; w < nw; ++w)
        for (int64_t p = window_row_ptr[w]; p < window_row_ptr[w + 1]; ++p) {
            int32_t col = window_col_idx[p];
            if (col < 0) continue;
            for (int64_t r = 0; r < h; ++r) {
                int64_t i = w * h + r;
                if (i >= m) break;
                double a = tab[values[r * P + p]];
                for (int64_t q = 0; q < n; ++q) C[i * n + q] += a * tab[B[(int64_t)col * n + q]];
            }
        }
    free(tab);
}

/* Number of threads an OpenMP parallel region uses here. */
int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
