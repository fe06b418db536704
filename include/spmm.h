/*
 * spmm.h -- C ABI of the GB300 (sm_103a) sparse x dense matrix multiply
 * library: C = A * B with A sparse (m x k), B dense (k x N, row-major) and
 * C dense (m x N, row-major), after "AsyncSparse: Accelerating Sparse
 * Matrix-Matrix Multiplication on Asynchronous GPU Architectures"
 * (Liu, Pu, Zhang).
 *
 * Two storage formats of A are offered, both from Section II-C and Fig. 2:
 *   BCSR  A cut into b_row x b_col blocks; blocks holding a nonzero are kept
 *         dense.  For block sparsity (Section III-C, Fig. 4).
 *   WCSR  rows grouped into windows of b_row rows; a window keeps the union
 *         of its rows' column indices (padded with -1 to a multiple of b_col)
 *         and a packed dense [b_row x columns] value tile.  For irregular
 *         sparsity (Sections II-C and III-B/C).
 *
 * Handles are created from a host CSR (the formats are built on the host and
 * uploaded), then run any number of times against device-resident B and C.
 *
 * Ownership: pointers passed to *_create are borrowed for the call only.  A
 * handle owns its device copies of the format, its task list and its split
 * workspace; spmm_destroy frees them.  B and C passed to spmm_run are
 * caller-owned device memory.  A handle must not be used by two host threads
 * at once; runs of one handle on different streams must not overlap on the
 * GPU (they share the split workspace).
 *
 * Errors: every call returns an spmm_status; spmm_last_error() gives a
 * message for the last failure on the calling thread.  spmm_run is
 * asynchronous and only reports launch-time errors; errors detected on the
 * device (a bounded wait that ran out, an index check) are recorded in a
 * status word that spmm_check reads.
 */
#ifndef SPMM_GB300_H
#define SPMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spmm_handle_s *spmm_handle;

typedef enum {
    SPMM_OK = 0,
    SPMM_ERR_INVALID_ARG = 1,  /* bad CSR, null pointer, bad size */
    SPMM_ERR_UNSUPPORTED = 2,  /* valid but not handled (N % 8, alignment, no sm_103 GPU ...) */
    SPMM_ERR_CUDA = 3,         /* a CUDA runtime / driver call failed */
    SPMM_ERR_OOM = 4,          /* device or host allocation failed */
    SPMM_ERR_TIMEOUT = 5,      /* a bounded wait inside a kernel ran out */
    SPMM_ERR_DEVICE_CHECK = 6  /* a kernel's own index check failed */
} spmm_status;

typedef enum { SPMM_F16 = 0, SPMM_BF16 = 1, SPMM_F32 = 2 } spmm_dtype;

typedef enum { SPMM_FORMAT_BCSR = 0, SPMM_FORMAT_WCSR = 1 } spmm_format;

/* Work schedule of the BCSR kernel (spmm_set_schedule). */
typedef enum {
    SPMM_SCHEDULE_AUTO = 0,   /* the library's choice (the default) */
    SPMM_SCHEDULE_TILES = 1,  /* whole tiles (block row x column tile) per CTA, round-robin */
    SPMM_SCHEDULE_SPLIT = 2,  /* equal shares of the tiles' stages per CTA; cut tiles summed by a second pass */
    SPMM_SCHEDULE_DYNAMIC = 3 /* WCSR: chunks of the work list taken over at run time (cluster launch control) */
} spmm_schedule;

/* Statistics of a handle's format (spmm_format_info). */
typedef struct {
    int32_t format;          /* spmm_format */
    int32_t b_row, b_col;    /* block rows x cols (BCSR); window height, column padding (WCSR) */
    int64_t m, k, nnz;
    int64_t n_groups;        /* block rows (BCSR) or windows (WCSR): ceil(m / b_row) */
    int64_t n_units;         /* stored blocks (BCSR) or padded column positions P_total (WCSR) */
    int64_t stored;          /* stored values: n_units*b_row*b_col (BCSR), b_row*P_total (WCSR) */
    int64_t padding;         /* stored - nnz: explicit zeros kept by the format */
    int64_t idx_bytes;       /* bytes of the index arrays on the device (ptr + idx) */
    int64_t val_bytes;       /* bytes of the value array on the device */
    int64_t n_tasks;         /* WCSR: stages (<= 64 packed columns of one window); BCSR: n_groups */
    int64_t n_split_windows; /* WCSR: windows cut between CTAs at N <= 256; BCSR: 0 */
    int64_t split_cols;      /* WCSR: packed columns per stage (64); BCSR: 0 */
} spmm_info;

/*
 * spmm_bcsr_create -- build a BCSR handle from a host CSR.
 * Paper: Section II-C "Block Compressed Sparse Row" and Fig. 2.  A block
 * (b_row x b_col) is kept iff it holds at least one CSR entry; kept blocks are
 * ordered by ascending block column within each block row and stored dense,
 * row-major, zero-filled.  The number of block rows is ceil(m / b_row).
 *   out       receives the handle (set to NULL on failure).
 *   m, k      A's shape, 0 <= m, k < 2^31.
 *   row_ptr   host int64[m+1], row_ptr[0] = 0, non-decreasing.
 *   col_idx   host int32[row_ptr[m]], each in [0, k), strictly ascending per row.
 *   vals      host 16-bit values (in_t bits), row_ptr[m] of them.  Every entry
 *             is structural: an explicit 0 still keeps its block.
 *   in_t      SPMM_F16 or SPMM_BF16 (type of A and of B at run time).
 *   out_t     SPMM_F32 or SPMM_BF16 (type of C); accumulation is fp32.
 *   b_row, b_col  block shape, 1..256 each.  spmm_run needs 64 x 64.
 * Errors: INVALID_ARG for a bad CSR or shape; OOM; CUDA (no device, upload).
 */
spmm_status spmm_bcsr_create(spmm_handle *out, int64_t m, int64_t k, const int64_t *row_ptr,
                             const int32_t *col_idx, const void *vals, spmm_dtype in_t,
                             spmm_dtype out_t, int b_row, int b_col);

/*
 * spmm_wcsr_create -- build a WCSR handle from a host CSR.
 * Paper: Section II-C "Window Compressed Sparse Row" and Fig. 2.  Window w
 * covers rows [w*window_h, (w+1)*window_h); its column list is the ascending
 * union of those rows' columns followed by -1 entries up to a multiple of
 * col_pad; window_row_ptr counts padded positions.  Values are one row-major
 * array [window_h][P_total]: element (r, p) is A[window_h*w + r][col(p)] for
 * the window w owning position p, 0 where absent or padded.
 * Arguments as for spmm_bcsr_create; window_h and col_pad in 1..256.
 * spmm_run takes window_h == 16 with col_pad a multiple of 16 (the window
 * rows are the N = 16 operand of a transposed MMA), or window_h == 64 with
 * col_pad a multiple of 8 (the paper's geometry, Section IV-A: the window rows
 * are the M = 64 operand); other shapes are rejected by spmm_run.
 * Windows are cut into stages of at most 64 packed columns; each persistent
 * CTA takes an equal number of stages (see spmm_set_max_ctas).
 */
spmm_status spmm_wcsr_create(spmm_handle *out, int64_t m, int64_t k, const int64_t *row_ptr,
                             const int32_t *col_idx, const void *vals, spmm_dtype in_t,
                             spmm_dtype out_t, int window_h, int col_pad);

/*
 * spmm_run -- C = A * B on the GPU, enqueued on `stream` (a cudaStream_t;
 * NULL = the legacy default stream).  Paper: BCSR kernel Section III-C
 * (Fig. 4), WCSR kernel Sections III-B/III-C.
 *   B  device pointer, k x N row-major, in_t, 16-byte aligned.
 *   C  device pointer, m x N row-major, out_t, 16-byte aligned; fully
 *      overwritten (rows of A without entries give 0).
 *   N  number of columns of B and C, N > 0 and N % 8 == 0 (TMA row stride).
 * A WCSR handle (and a BCSR one on the split schedule) adds the partial sums
 * of groups cut between CTAs in a second kernel, in a fixed order, using a
 * workspace allocated at create; results are bitwise reproducible run to run.
 * That kernel is launched as a programmatic dependent of the first (it may
 * be scheduled before the first finishes and waits for it on the device);
 * to the caller the two behave as one stream-ordered operation, also under
 * stream capture.
 * Errors: INVALID_ARG (null handle/pointers, N <= 0); UNSUPPORTED (N % 8,
 * alignment, format parameters the kernels do not take, device not sm_103);
 * OOM (workspace); CUDA (launch).  Asynchronous: see spmm_check.
 */
spmm_status spmm_run(spmm_handle h, const void *B, void *C, int64_t N, void *stream);

/*
 * spmm_run_linear -- Y = X * A^T for a BCSR handle with 64 x 64 blocks: the
 * product in the layout of a linear layer whose weight is A (m output
 * features x k input features), Y[n][i] = sum_j X[n][j] * A[i][j].  X is the
 * dense operand B = X^T of C = A * B stored column-major, the layout the
 * paper's BCSR kernel reads B in (Section III-B) and the one of its drop-in
 * replacement of a linear layer (Section IV-D, Table III); Y = C^T.
 *   X  device pointer, N x k row-major, in_t, 16-byte aligned; k % 8 == 0.
 *   Y  device pointer, N x m row-major, out_t, 16-byte aligned, fully
 *      overwritten; m % 8 == 0 for bf16 Y, m % 4 == 0 for fp32 Y.
 *   N  rows of X and Y (tokens), N > 0; no multiple is required.
 * Asynchronous on `stream`; errors as spmm_run, plus UNSUPPORTED for a WCSR
 * handle.  Rows of X are read by 256-row tiles; results are bitwise
 * reproducible run to run.
 */
spmm_status spmm_run_linear(spmm_handle h, const void *X, void *Y, int64_t N, void *stream);

/*
 * spmm_run_host -- the same product with B and C in HOST memory: copies B to
 * the device, runs, copies C back, all on `stream`, and waits for the stream.
 * Device staging buffers are owned by the handle and grow on demand.  Pinned
 * host memory gives the fastest copies.  Errors as spmm_run, plus device
 * errors recorded by the kernels (it calls spmm_check).
 */
spmm_status spmm_run_host(spmm_handle h, const void *B_host, void *C_host, int64_t N, void *stream);

/* spmm_destroy -- free the handle and its device memory (waits for the device). */
spmm_status spmm_destroy(spmm_handle h);

/* spmm_format_info -- statistics of the handle's format, written to *info. */
spmm_status spmm_format_info(spmm_handle h, spmm_info *info);

/*
 * spmm_export_format -- host copies of the three format arrays, for
 * comparison with an independent converter.
 *   ptr_out   int64[n_groups + 1]   block_row_ptr / window_row_ptr
 *   idx_out   int32[n_units]        block_col_idx / window_col_idx (-1 = padding)
 *   vals_out  uint16[stored]        blocks (n_units x b_row x b_col) / values (b_row x P_total)
 * Any of the three may be NULL to skip it.
 */
spmm_status spmm_export_format(spmm_handle h, int64_t *ptr_out, int32_t *idx_out, uint16_t *vals_out);

/*
 * spmm_bcsr_convert -- host-only CSR -> BCSR with the converter that
 * spmm_bcsr_create uses (no GPU needed).  Paper: Section II-C and Fig. 2.
 * Call once with block_col_idx == NULL to get *n_blocks, then again with
 *   block_row_ptr  int64[ceil(m/b_row) + 1]
 *   block_col_idx  int32[*n_blocks]
 *   blocks         uint16[*n_blocks * b_row * b_col] (may be NULL: skip values)
 * Errors: INVALID_ARG for a bad CSR or shape.
 */
spmm_status spmm_bcsr_convert(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                              const void *vals, int b_row, int b_col, int64_t *n_blocks,
                              int64_t *block_row_ptr, int32_t *block_col_idx, uint16_t *blocks);

/*
 * spmm_wcsr_convert -- host-only CSR -> WCSR with the converter that
 * spmm_wcsr_create uses.  Paper: Section II-C and Fig. 2.  Call once with
 * window_col_idx == NULL to get *p_total, then again with
 *   window_row_ptr  int64[ceil(m/window_h) + 1]
 *   window_col_idx  int32[*p_total]  (-1 = padding)
 *   values          uint16[window_h * *p_total] row-major (may be NULL)
 * Errors: INVALID_ARG for a bad CSR or shape.
 */
spmm_status spmm_wcsr_convert(int64_t m, int64_t k, const int64_t *row_ptr, const int32_t *col_idx,
                              const void *vals, int window_h, int col_pad, int64_t *p_total,
                              int64_t *window_row_ptr, int32_t *window_col_idx, uint16_t *values);

/*
 * spmm_check -- wait for `stream`, then read and clear the handle's device
 * status word.  Returns SPMM_ERR_TIMEOUT if a kernel's bounded wait ran out,
 * SPMM_ERR_DEVICE_CHECK if a kernel's index check failed, SPMM_ERR_CUDA for a
 * sticky CUDA error, else SPMM_OK.
 */
spmm_status spmm_check(spmm_handle h, void *stream);

/*
 * spmm_set_max_ctas -- cap the number of persistent CTAs a run launches
 * (ctas = 0, the default: two CTAs per SM for WCSR with 16-row windows, one
 * with 64-row windows; for BCSR one per SM, or two per SM when N > 128 and
 * there are at least two 256-column tiles per SM; WCSR caps ctas at two per
 * SM).  Under the WCSR dynamic schedule the cap sets the CTAs that fit, and
 * the grid holds about four chunks per such CTA.  Both kernels give each CTA an equal
 * share of the work (BCSR: whole block-row x column tiles; WCSR: equal
 * numbers of 64-column stages), so the cap changes where WCSR windows are cut
 * between CTAs (their partial sums are added by a second kernel in a fixed
 * order) but not the result beyond fp32 rounding.
 */
spmm_status spmm_set_max_ctas(spmm_handle h, int32_t ctas);

/*
 * spmm_set_schedule -- choose how a handle's spmm_run spreads work over CTAs.
 * BCSR handles: SPMM_SCHEDULE_TILES gives each persistent CTA whole tiles (one
 * block row x one tile of 128 or 256 columns), as the paper's static grid
 * does (Section III-F).  SPMM_SCHEDULE_SPLIT lists the stages of all tiles
 * (one per stored block; one for a block row without blocks) and gives each
 * CTA an equal contiguous share, so long block rows are spread over several
 * CTAs (the load balance that the paper's WCSR task decomposition gives
 * windows, Section III-C); tiles cut between CTAs leave fp32 partial sums
 * that a second kernel adds in CTA order, so results stay bitwise
 * reproducible.  SPMM_SCHEDULE_AUTO (the default) takes the split schedule
 * only when fewer than half the SMs would get a tile and the tiles average at
 * least 8 stages.  The split schedule needs a handle with fewer than two block
 * rows per SM (its workspace is allocated at create only then); otherwise
 * SPLIT runs as TILES.
 * WCSR handles with window height 16: AUTO, TILES and SPLIT all give each
 * persistent CTA an equal contiguous share of the work items (stages x column
 * tiles).  SPMM_SCHEDULE_DYNAMIC cuts the work list into about four times as
 * many chunks as CTAs fit on the GPU (each of at least 32 items) and launches
 * one CTA per chunk; a running CTA that finishes a chunk cancels the launch of
 * a CTA that has not started and takes over its chunk (cluster launch
 * control, the dynamic scheduling the paper names as future work for
 * Blackwell, Section V), so faster CTAs take more chunks.  Windows cut
 * between chunks are summed in chunk order by the second kernel, so results
 * do not depend on which CTA ran which chunk.  Setting DYNAMIC allocates the
 * larger partial-sum workspace it needs (about 40 MB at 152 SMs).
 * Errors: INVALID_ARG (null handle, unknown schedule); UNSUPPORTED (DYNAMIC on
 * a BCSR handle or a WCSR handle whose windows are not 16 rows high); OOM.
 */
spmm_status spmm_set_schedule(spmm_handle h, int32_t schedule);

/*
 * spmm_selftest_wait_timeout -- failure-detection self test.  Launches one
 * CTA whose thread waits on an mbarrier that nothing arrives at, with a limit
 * of timeout_ns nanoseconds, through the same bounded-wait routine the SpMM
 * kernels use; the kernel then records a timeout and returns.  Waits for the
 * stream and returns the recorded status in *dev_status (SPMM_ERR_TIMEOUT
 * when the bound works).  timeout_ns must be in [1000, 10^10].
 */
spmm_status spmm_selftest_wait_timeout(int64_t timeout_ns, void *stream, int32_t *dev_status);

/*
 * spmm_probe_l2_read -- measurement helper, not part of the product: reads
 * `bytes` of device memory at `buf`, `passes` times, with 16-byte loads that
 * bypass L1, from four CTAs of 512 threads per SM, enqueued on `stream`.  With
 * a buffer that stays in L2 (a few tens of MB) and one untimed pass first,
 * the caller's CUDA-event time gives the L2-to-SM read rate, the ceiling of
 * the WCSR gather, which fetches rows of an L2-resident B by index
 * (Section III-B).
 *   buf    device pointer, 16-byte aligned; bytes > 0 and a multiple of 16.
 *   sink   device pointer to 16 writable bytes; written only when the XOR of
 *          the data read equals a fixed constant (it keeps the loads alive).
 * Errors: INVALID_ARG (null pointers, bytes, passes < 1, alignment); CUDA
 * (launch).  Asynchronous.
 */
spmm_status spmm_probe_l2_read(const void *buf, int64_t bytes, int32_t passes, void *sink, void *stream);

/*
 * spmm_wcsr_run_noalloc -- C = A * B for A in WCSR, for callers that cannot
 * allocate device memory when they run the product: code whose device memory
 * all comes from its own pool or arena, or which must not call cudaMalloc /
 * cudaFree at that point (they may synchronise the device).  The paper has
 * no counterpart; it runs the same WCSR kernel as spmm_run.
 * The caller passes device arrays of a WCSR format with window height 16 and
 * a column padding that is a multiple of 16 (as spmm_wcsr_create /
 * spmm_export_format produce them):
 *   window_row_ptr  int64[ceil(m/16) + 1]
 *   window_col_idx  int32[p_total]       (-1 = padding; other entries in [0, k))
 *   values          16-bit [16][p_total] row-major, in_t, 16-byte aligned
 * and B (k x N) and C (m x N) as for spmm_run; C is fully overwritten.
 * Nothing is allocated: the work list and the partial sums of windows cut
 * between CTAs live in one static device array of about 10 MB that every GPU
 * which loads this library holds until the process exits.  Its limit:
 * ceil(m/16) + p_total/64 <= 131072; larger problems are rejected with
 * SPMM_ERR_UNSUPPORTED before anything is launched.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress), so make
 * that first call before any stream capture on that device.
 * Every call uses the same array, which keeps the previous call's contents
 * (each call rebuilds what it reads): calls whose work overlaps on the GPU
 * (other streams, other host threads) race and must be serialised by the
 * caller.  Asynchronous on `stream`; a bounded wait that runs out, or a
 * window_row_ptr that fails the device-side check (first entry 0, entries
 * non-decreasing multiples of 16, last entry p_total), is reported by
 * spmm_wcsr_noalloc_check, not here.
 * Errors: INVALID_ARG (null pointers, sizes), UNSUPPORTED (N % 8,
 * alignment, p_total % 16, the size limit, no sm_103 device), CUDA (launch).
 */
spmm_status spmm_wcsr_run_noalloc(const int64_t *window_row_ptr, const int32_t *window_col_idx,
                                  const void *values, int64_t m, int64_t k, int64_t p_total,
                                  spmm_dtype in_t, spmm_dtype out_t, const void *B, void *C,
                                  int64_t N, void *stream);

/*
 * spmm_wcsr_noalloc_check -- waits for `stream`, then reads and clears the
 * status word that spmm_wcsr_run_noalloc calls on the current device share
 * (a call resets it when it starts, so it describes the last call):
 * SPMM_OK; SPMM_ERR_DEVICE_CHECK when window_row_ptr failed the device-side
 * check (no work was listed, C was left as it was); SPMM_ERR_TIMEOUT when a
 * bounded wait ran out (C is incomplete).  Allocates nothing.
 * Errors: CUDA (the copy or the synchronisation).
 */
spmm_status spmm_wcsr_noalloc_check(void *stream);

/* spmm_status_str -- static English name of a status. */
const char *spmm_status_str(spmm_status s);

/* spmm_last_error -- message for the last failing call on this thread ("" if none). */
const char *spmm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPMM_GB300_H */
