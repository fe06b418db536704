// internal.h -- launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace spmm {

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: the attribute is held per device, so a process
// that runs on several GPUs sets it on each.  `done` holds one bit per device
// ordinal (below 64; others set it on every call).  Two host threads may both
// set it; the call is idempotent.
template <typename Kernel>
cudaError_t set_smem_limit_once(Kernel kern, int bytes, std::atomic<uint64_t> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Flags of a stage / segment: it holds the first and/or the last stage of its
// group (a WCSR window, or a BCSR block row x column tile).
constexpr int32_t kStageFirst = 1;
constexpr int32_t kStageLast = 2;

// A partial sum written to a split workspace by a persistent CTA whose share
// of stages cuts a group: the group (WCSR window or BCSR block row), its
// column tile and whether it holds the group's first and/or last stage.
struct PartialRec {
  int32_t group;     // -1: slot unused in this run
  int32_t col_tile;
  int32_t flags;     // kStageFirst | kStageLast
  int32_t pad_;
};

// BCSR SpMM.  Work unit ("tile") = one block row x one tile of N columns.
// Default schedule: persistent CTAs take whole tiles round-robin.  Split
// schedule (split_grid > 0, for problems with fewer tiles than about two per
// SM): the tiles' stages (one per stored block, one for a block row without
// blocks) are listed tile after tile and CTA c takes the equal contiguous
// share [T*c/G, T*(c+1)/G); tiles cut between CTAs leave fp32 partial sums
// that split_reduce_kernel adds in CTA order.
struct BcsrParams {
  const int64_t *block_row_ptr;  // device, n_block_rows + 1
  const int32_t *block_col_idx;  // device, n_blocks
  const void *blocks;            // device, n_blocks x 64 x 64 row-major
  const int64_t *stage_row_ptr;  // device, n_block_rows + 1: prefix sums of max(1, blocks of the block row)
  const void *B;                 // device, K x N row-major
  void *C;                       // device, M x N row-major
  float *workspace;              // split schedule: 2 slots per CTA of 64 x 256 fp32
  PartialRec *partials;          // split schedule: 2 records per CTA
  int64_t ldc;                   // row stride of C in elements (= N)
  int32_t M, N, K;
  int32_t n_block_rows;
  int32_t max_ctas;              // cap on the persistent grid (0: the kernel's default CTAs per SM)
  int32_t num_sms;
  int32_t split_grid;            // > 0: split schedule over this many CTAs
  int64_t split_stages;          // split schedule: stages per column tile (stage_row_ptr[n_block_rows])
  int64_t n_blocks;              // stored blocks (block_row_ptr[n_block_rows])
  uint32_t *status;              // device status word
  uint64_t wait_limit_ns;        // bound of every mbarrier wait
};

// Split-schedule workspace: floats per slot (64 rows x 256 columns) and the
// largest grid it is sized for, in CTAs per SM.
constexpr int64_t kBcsrSlotFloats = 64 * 256;
constexpr int kBcsrSplitCtasPerSm = 2;
// The split schedule is used when the tiles number fewer than this many per
// SM, and gives each CTA at least kBcsrSplitMinStages stages.
constexpr int kBcsrSplitBelowTilesPerSm = 2;
constexpr int kBcsrSplitMinStages = 4;

// The BCSR kernel's C store boxes: for N <= 128, 16 rows x 128 bytes with the
// 128-byte swizzle; wider, 32 rows x 64 bytes with the 64-byte swizzle.
inline bool bcsr_wide_tiles(int64_t N) { return N > 128; }
// Columns of C per BCSR tile at dense width N (256 for wide tiles, else 128).
int bcsr_tile_cols(int64_t N);

// in_bf16: A/B are bf16 (else fp16); out_bf16: C is bf16 (else fp32).
// tmA covers the blocks array as [n_blocks*64 rows, 64 cols], tmB covers B as
// [K rows, N cols]; both with 64 x 64 boxes and 128-byte swizzle.  tmC covers
// C as [M rows, N cols] with the boxes of bcsr_wide_tiles(N).
cudaError_t launch_bcsr(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const BcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t stream);

// BCSR product in the layout of a linear layer, Y = X * A^T (bcsr_linear_kernel.cu):
// p.B is X (N x K row-major), p.C is Y (N x M row-major).  tmA covers the
// blocks as for launch_bcsr; tmX covers X as [N rows, K cols] with 256-row x
// 64-column boxes, 128-byte swizzle; tmY covers Y as [N rows, M cols] with
// 32-row x 128-byte boxes, 128-byte swizzle.
cudaError_t launch_bcsr_linear(const CUtensorMap &tmA, const CUtensorMap &tmX, const CUtensorMap &tmY,
                               const BcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t stream);

// WCSR work is a list of stages: at most 64 packed columns of one window.
// Every window has at least one stage (ncols = 0 for a window without
// columns), and stages are listed in window order.
struct WcsrStage {
  int32_t p_begin;   // first packed column
  int32_t window;
  int32_t ncols;     // 0..64, a multiple of 16
  int32_t flags;     // kStageFirst | kStageLast
};

// One stage as a record of kWcsrPackBytes in device memory, fetched by one
// TMA bulk copy: the 16 x 64 value tile in the MMA's swizzled K-major layout
// (zero past ncols), the 64 column indices (-1 for a padding position, -2
// past ncols) and the descriptor {ncols, flags, window, 0}.
constexpr int kWcsrPackValOff = 0;
constexpr int kWcsrPackIdxOff = 2048;
constexpr int kWcsrPackDescOff = 2048 + 256;
constexpr int kWcsrPackBytes = 2048 + 256 + 16;
// The same record for a window of h rows (16 or 64): an h x 64 value tile,
// then the 64 indices and the descriptor.
constexpr int wcsr_pack_idx_off(int h) { return h * 64 * 2; }
constexpr int wcsr_pack_desc_off(int h) { return h * 64 * 2 + 256; }
constexpr int wcsr_pack_bytes(int h) { return h * 64 * 2 + 256 + 16; }
static_assert(wcsr_pack_bytes(16) == kWcsrPackBytes && wcsr_pack_bytes(64) % 16 == 0, "record layout");

#ifdef __CUDACC__
// Work item f of a WCSR grid is (column tile f / n_stages, stage record
// f % n_stages).  A producer walks its items in small increasing steps, so
// the cursor follows them with additions and divides only when f jumps (a
// 64-bit division is a long instruction sequence on the GPU).
struct ItemCursor {
  int64_t f = -1;  // current item
  int64_t s = 0;   // its stage record
  int tile = 0;    // its column tile
  __device__ __forceinline__ void to(int64_t nf, int64_t n_stages) {
    if (f < 0 || nf < f || nf - f > n_stages) {
      tile = static_cast<int>(nf / n_stages);
      s = nf - static_cast<int64_t>(tile) * n_stages;
    } else {
      s += nf - f;
      while (s >= n_stages) {
        s -= n_stages;
        ++tile;
      }
    }
    f = nf;
  }
};
#endif

struct WcsrParams {
  const WcsrStage *stages;       // device, n_stages (the no-allocation variant's stage list)
  const void *stage_pack;        // device, n_stages x kWcsrPackBytes (the allocating entry points)
  const void *values;            // device, 16 x P_total row-major (read by the no-allocation variant)
  const int32_t *window_col_idx; // device, P_total (read by the no-allocation variant only)
  const int64_t *n_stages_dev;   // device stage count (no-allocation variant only)
  const void *B;                 // device, K x N row-major
  void *C;                       // device, M x N row-major
  float *workspace;              // device, 2 * grid x 16 x 256 fp32
  PartialRec *partials;          // device, 2 * grid
  int64_t n_stages;
  int64_t P_total;
  int32_t M, N, K;
  int32_t grid;                  // CTAs launched = chunks: chunk c is a contiguous range of (column tile, stage)
  int32_t dynamic;               // window height 16: running CTAs take over chunks of CTAs not yet started
  uint32_t *status;
  uint64_t wait_limit_ns;
};

// Persistent WCSR CTAs per SM at dense width N (the default grid is this
// times the SM count), and the most it can be (the partial-sum workspace is
// sized for it).
int wcsr_ctas_per_sm(int64_t N);
// Columns of C per WCSR work item (window height 16) at dense width N.
int wcsr_tile_cols(int64_t N);
constexpr int kWcsrMaxCtasPerSm = 2;
// Dynamic WCSR schedule: chunks per CTA that fits on the GPU, and the fewest
// work items a chunk may hold.
constexpr int kWcsrDynChunksPerCta = 4;
constexpr int64_t kWcsrDynMinChunkItems = 32;

// Workspace floats per partial slot (16 rows x 256 columns).
constexpr int64_t kWcsrSlotFloats = 16 * 256;

// Limits of spmm_wcsr_run_noalloc's static scratch.
constexpr int64_t kNoallocMaxStages = 131072;
constexpr int kNoallocMaxCtas = 256;

// spmm_wcsr_run_noalloc's launches: builds the stage list from the caller's
// window_row_ptr into the static scratch, runs the WCSR kernel's no-allocation
// variant and the partial-sum pass.  p carries the caller's arrays, B, C and
// the sizes; the scratch pointers are filled in here.
// Copies the no-allocation scratch's status word of the current device into
// *word and clears it, after the work queued on `stream` (synchronises it).
cudaError_t wcsr_noalloc_take_status(uint32_t *word, cudaStream_t stream);
cudaError_t launch_wcsr_noalloc(WcsrParams p, const int64_t *window_row_ptr, int64_t n_windows, int num_sms,
                                bool in_bf16, bool out_bf16, cudaStream_t stream);
size_t wcsr_noalloc_scratch_bytes();

// Runs the SpMM kernel, then the kernel that adds the partials of windows
// cut between CTAs.
cudaError_t launch_wcsr(const WcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t stream);

// WCSR with 64-row windows (wcsr64_kernel.cu): stage records of
// wcsr_pack_bytes(64), 256-column tiles, whole windows stored through tmC
// (C as [M rows, N cols], 32-row x 64-byte boxes, 64-byte swizzle), windows
// cut between CTAs as 64 x 256 fp32 partials (kWcsr64SlotFloats per slot)
// added by split_reduce_kernel.
constexpr int64_t kWcsr64SlotFloats = 64 * 256;
int wcsr64_ctas_per_sm();
cudaError_t launch_wcsr64(const CUtensorMap &tmC, const WcsrParams &p, bool in_bf16, bool out_bf16,
                          cudaStream_t stream);

// Failure-detection self test: wait on an mbarrier nothing arrives at.
cudaError_t launch_wait_selftest(uint32_t *status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace spmm
