// internal.h -- launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spmm {

// BCSR SpMM: one CTA per (block row, tile of N columns).
struct BcsrParams {
  const int64_t *block_row_ptr;  // device, n_block_rows + 1
  const int32_t *block_col_idx;  // device, n_blocks
  const void *blocks;            // device, n_blocks x 64 x 64 row-major
  const void *B;                 // device, K x N row-major
  void *C;                       // device, M x N row-major
  int64_t ldc;                   // row stride of C in elements (= N)
  int32_t M, N, K;
  int32_t n_block_rows;
  int32_t max_ctas;              // persistent grid size (one CTA per SM)
  uint32_t *status;              // device status word
  uint64_t wait_limit_ns;        // bound of every mbarrier wait
};

// in_bf16: A/B are bf16 (else fp16); out_bf16: C is bf16 (else fp32).
// tmA covers the blocks array as [n_blocks*64 rows, 64 cols], tmB covers B as
// [K rows, N cols]; both with 64 x 64 boxes and 128-byte swizzle.
cudaError_t launch_bcsr(const CUtensorMap &tmA, const CUtensorMap &tmB, const BcsrParams &p, bool in_bf16,
                        bool out_bf16, cudaStream_t stream);

// WCSR task: packed columns [p_begin, p_end) of one window.
struct WcsrTask {
  int32_t window;
  int32_t slot;      // -1: the task covers the whole window and writes C; else partial index
  int64_t p_begin;
  int64_t p_end;
};

// A window split across several tasks: its partials are slots
// [slot_begin, slot_begin + n_slots), summed in that order.
struct WcsrSplit {
  int32_t window;
  int32_t slot_begin;
  int32_t n_slots;
  int32_t pad_;
};

struct WcsrParams {
  const WcsrTask *tasks;         // device, n_tasks
  const int32_t *window_col_idx; // device, P_total
  const void *B;                 // device, K x N row-major
  void *C;                       // device, M x N row-major
  float *workspace;              // device, n_slots x 16 x N fp32 (split windows only)
  int64_t P_total;
  int32_t M, N, K;
  int32_t n_tasks;
  uint32_t *status;
  uint64_t wait_limit_ns;
};

// tmV covers the values array as [16 rows, P_total cols] with 64 x 16 boxes;
// tmB covers B as [K rows, N cols] with 64 x 1 boxes (row gathers); both with
// 128-byte swizzle.
cudaError_t launch_wcsr(const CUtensorMap &tmV, const CUtensorMap &tmB, const WcsrParams &p, bool in_bf16,
                        bool out_bf16, cudaStream_t stream);

// Sum the partials of split windows into C in slot order.
cudaError_t launch_wcsr_reduce(const WcsrSplit *splits, int32_t n_splits, const float *workspace,
                               void *C, int32_t M, int32_t N, bool out_bf16, cudaStream_t stream);

// Failure-detection self test: wait on an mbarrier nothing arrives at.
cudaError_t launch_wait_selftest(uint32_t *status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace spmm
