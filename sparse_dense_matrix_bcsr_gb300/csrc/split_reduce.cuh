// split_reduce.cuh -- second pass of the equal-share schedules: adds the fp32
// partial sums of the groups (a WCSR window, or a BCSR block row x column
// tile) whose stages were cut between persistent CTAs, in CTA order, and
// writes the group's rows of C.
//
// The paper adds such partials with atomicAdd ("AsyncSparse", Section III-C);
// summing the slots in a fixed order instead makes every run bitwise equal.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace spmm {

template <bool OUT_BF16>
__device__ __forceinline__ void store_out(void *C, int64_t off, float v) {
  if constexpr (OUT_BF16)
    reinterpret_cast<__nv_bfloat16 *>(C)[off] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float *>(C)[off] = v;
}

// Block (b, y) handles slot b, rows [y * RPB, (y + 1) * RPB) of its group.
// Slot 2c holds CTA c's first segment (the one that starts at the first stage
// of its share), slot 2c + 1 its last; a slot whose record has kStageFirst
// but not kStageLast starts a cut group: its blocks add it and the
// first-segment slots of the following CTAs, in CTA order, until the one
// whose record has kStageLast, and write the group's rows of C (ROWS x bn
// values at rows ROWS * group, columns bn * col_tile).  Slot s holds rows at
// ws + s * slot_floats + row * ws_ld.  The first warp finds the contributing
// slots 32 records at a time (dynamic shared memory, one int per CTA of the
// first pass); each thread then sums four adjacent columns, every load
// independent of the others, so the pass costs a few memory latencies.
template <int ROWS, int RPB, bool OUT_BF16>
__global__ void __launch_bounds__(256)
    split_reduce_kernel(const PartialRec *partials, const float *ws, int64_t slot_floats, int32_t ws_ld, void *C,
                        int32_t M, int32_t N, int32_t grid, int32_t bn) {
  static_assert(ROWS % RPB == 0, "row chunks");
  extern __shared__ int32_t contrib[];  // [grid]
  __shared__ int32_t n_contrib;
  grid_dependency_wait();  // the first pass has finished and its partials are visible
  const int slot = blockIdx.x;
  const PartialRec rec = partials[slot];
  if (rec.group < 0 || !(rec.flags & kStageFirst) || (rec.flags & kStageLast)) return;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int n = 1;
    if (lane == 0) contrib[0] = slot;
    for (int c0 = slot / 2 + 1; c0 < grid; c0 += 32) {
      const int c = c0 + lane;
      PartialRec r{-1, 0, 0, 0};
      if (c < grid) r = partials[2 * c];
      const bool same = c < grid && r.group == rec.group && r.col_tile == rec.col_tile;
      const unsigned not_same = __ballot_sync(0xffffffffu, !same);
      const unsigned last = __ballot_sync(0xffffffffu, same && (r.flags & kStageLast));
      const int stop = not_same ? __ffs(not_same) - 1 : 32;       // first lane outside the group
      const int end = last ? __ffs(last) : 32;                     // one past the first lane holding the last stage
      const int cnt = stop < end ? stop : end;
      if (lane < cnt) contrib[n + lane] = 2 * c;
      n += cnt;
      if (cnt < 32 || last) break;
    }
    if (lane == 0) n_contrib = n;
  }
  __syncthreads();
  const int n = n_contrib;
  const int n0 = rec.col_tile * bn;
  const int width = min(bn, N - n0);  // a multiple of 8 (N is)
  const int r0 = blockIdx.y * RPB;
  for (int e = 4 * threadIdx.x; e < RPB * width; e += 4 * blockDim.x) {
    const int q = r0 + e / width;
    const int col = e - (q - r0) * width;  // a multiple of 4
    const int row = rec.group * ROWS + q;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n; ++i) {
      const float4 v =
          *reinterpret_cast<const float4 *>(ws + static_cast<int64_t>(contrib[i]) * slot_floats + q * ws_ld + col);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (row < M) {
      const int64_t o = static_cast<int64_t>(row) * N + n0 + col;
      store_out<OUT_BF16>(C, o, acc.x);
      store_out<OUT_BF16>(C, o + 1, acc.y);
      store_out<OUT_BF16>(C, o + 2, acc.z);
      store_out<OUT_BF16>(C, o + 3, acc.w);
    }
  }
}

// Launches split_reduce_kernel over 2 * grid slots in chunks of 8 rows.
template <int ROWS, bool OUT_BF16>
inline cudaError_t launch_split_reduce(const PartialRec *partials, const float *ws, int64_t slot_floats,
                                       int32_t ws_ld, void *C, int32_t M, int32_t N, int32_t grid, int32_t bn,
                                       cudaStream_t stream) {
  constexpr int kRpb = 8;
  // Launched as a programmatic dependent of the first pass: its launch
  // overlaps the first pass's last tiles, and grid_dependency_wait holds its
  // blocks until the first pass has completed.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * grid, ROWS / kRpb);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = grid * sizeof(int32_t);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_reduce_kernel<ROWS, kRpb, OUT_BF16>, partials, ws, slot_floats, ws_ld, C,
                            M, N, grid, bn);
}

}  // namespace spmm
