// wcsr_kernel.cu -- WCSR SpMM for sm_103a.
//
// Method: "AsyncSparse", Section III-B (the packed value tile of a window is
// contiguous and loaded by TMA; the matching rows of B are fetched through
// window_col_idx) and Section III-C (task-based decomposition: long windows
// are split into fixed-size sub-tasks and the CTA index names a task).  On
// Hopper the paper gathers B with all threads of a warpgroup because TMA
// cannot gather; sm_103a's TMA can (tile::gather4, four rows per
// instruction), so here one producer warp issues every load, as in the BCSR
// kernel, and the MMA runs decoupled behind an mbarrier ring.  The paper adds
// split partial sums with atomicAdd; here a split task writes an fp32 partial
// and a second kernel adds a window's partials in slot order, so results are
// bitwise reproducible.
//
// The product is computed transposed: the 128 columns of an accumulator are
// the MMA's M (TMEM lanes) and the 16 rows of a window are the MMA's N, so a
// 16-row window is a legal tcgen05 shape.
//
// CTA = one task x one tile of BN = 128*NACC columns; 6 warps:
//   warp 0      producer: value tile (2-D TMA) and B rows (TMA gather4); the
//               warp prefetches the column indices PF stages ahead
//   warp 1      TMEM allocator and MMA issuer
//   warps 2..5  epilogue (warp w reads TMEM sub-partition w % 4)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace spmm {
namespace {

constexpr int kH = 16;                       // window height
constexpr int kKC = 64;                      // packed columns per stage
constexpr int kValBytes = kH * kKC * 2;      // 2 KB value tile per stage
constexpr int kChunkBytes = kKC * 64 * 2;    // 64 gathered rows x 64 columns
constexpr int kThreads = 192;
constexpr int kPF = 4;                       // index prefetch distance (stages)

template <int NACC, int Q>
struct Cfg {
  static constexpr int kBN = 128 * NACC;
  static constexpr int kChunks = 2 * NACC;
  static constexpr int kStageBytes = kValBytes + kChunks * kChunkBytes;
  static constexpr int kTmemCols = 32;  // NACC * 16 <= 32
  static constexpr int kSmemBytes = Q * kStageBytes + 1024 + 1024;
};

template <bool OUT_BF16>
__device__ __forceinline__ void store_out(void *C, int64_t off, float v) {
  if constexpr (OUT_BF16)
    reinterpret_cast<__nv_bfloat16 *>(C)[off] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float *>(C)[off] = v;
}

template <int NACC, int Q, bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    wcsr_spmm_kernel(const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmB,
                     const WcsrParams p) {
  using C_ = Cfg<NACC, Q>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Q * C_::kStageBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * Q + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WcsrTask task = p.tasks[blockIdx.x];
  const int n0 = blockIdx.y * C_::kBN;
  const int nvalid = min(C_::kBN, p.N - n0);
  const int nacc = min(NACC, (nvalid + 127) / 128);
  const int nch = min(C_::kChunks, (nvalid + 63) / 64);
  const int64_t ncols = task.p_end - task.p_begin;
  const int nstages = static_cast<int>((ncols + kKC - 1) / kKC);

  const uint32_t full0 = smem_addr(&bars[0]);
  const uint32_t empty0 = smem_addr(&bars[Q]);
  const uint32_t accum_bar = smem_addr(&bars[2 * Q]);
  const uint32_t drain_bar = smem_addr(&bars[2 * Q + 1]);

  if (threadIdx.x == 0) {
    for (int q = 0; q < Q; ++q) {
      mbar_init(full0 + 8 * q, 1);
      mbar_init(empty0 + 8 * q, 1);
    }
    mbar_init(accum_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C_::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane l gathers row group g = l % 16 (rows 4g..4g+3 of a stage) for the
    // column chunks of its half-warp.
    const int g = lane & 15;
    constexpr int kChunksPerLane = C_::kChunks / 2;
    const int c_first = (lane >> 4) * kChunksPerLane;
    const int32_t oob_row = p.K;  // padding (-1) gathers an out-of-range row: TMA fills zeros
    auto load_idx = [&](int s) -> int4 {
      const int64_t pb = task.p_begin + static_cast<int64_t>(s) * kKC + 4 * g;
      if (s < nstages && pb < task.p_end) return *reinterpret_cast<const int4 *>(p.window_col_idx + pb);
      return make_int4(-2, -2, -2, -2);
    };
    // Index prefetch ring: slot u holds the indices of stage s with s % kPF == u.
    // The loop is unrolled by kPF so every slot stays in a fixed register and a
    // load is only waited for when its stage is issued, kPF stages later.
    int4 ring[kPF];
#pragma unroll
    for (int i = 0; i < kPF; ++i) ring[i] = load_idx(i);

    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int s0 = 0; s0 < nstages && ok; s0 += kPF) {
#pragma unroll
      for (int u = 0; u < kPF; ++u) {
        const int s = s0 + u;
        if (s >= nstages || !ok) break;
        const int4 cur = ring[u];
        ring[u] = load_idx(s + kPF);

        if (lane == 0) ok = mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns) && !*abort_flag;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int64_t pbase = task.p_begin + static_cast<int64_t>(s) * kKC;
        const int64_t left = task.p_end - pbase;
        const int groups = left >= kKC ? kKC / 4 : static_cast<int>(left / 4);
        const uint32_t st = smem_addr(smem + stage * C_::kStageBytes);
        const uint32_t fb = full0 + 8 * stage;
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, kValBytes + groups * 4 * 128 * nch);
          tma_load_2d(st, &tmV, fb, static_cast<int32_t>(pbase), 0);
        }
        __syncwarp();
        if (g < groups) {
          const int32_t r0 = cur.x < 0 ? oob_row : cur.x;
          const int32_t r1 = cur.y < 0 ? oob_row : cur.y;
          const int32_t r2 = cur.z < 0 ? oob_row : cur.z;
          const int32_t r3 = cur.w < 0 ? oob_row : cur.w;
#pragma unroll
          for (int j = 0; j < kChunksPerLane; ++j) {
            const int c = c_first + j;
            if (c < nch)
              tma_gather4(st + kValBytes + c * kChunkBytes + g * 512, &tmB, fb, n0 + c * 64, r0, r1, r2, r3);
          }
        }
        ++issued;
        if (++stage == Q) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      atomicOr(p.status, kDevTimeout);
      *abort_flag = 1;
      const int64_t first = issued > Q ? issued - Q : 0;
      for (int64_t i = first; i < issued; ++i)
        mbar_wait(full0 + 8 * (i % Q), static_cast<uint32_t>((i / Q) & 1), 1000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nstages > 0) {
      constexpr uint32_t idesc = idesc_f16(IN_BF16, /*a_mn_major=*/true, /*b_mn_major=*/false, 128, kH);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int s = 0; s < nstages; ++s) {
        if (!mbar_wait(full0 + 8 * stage, phase, p.wait_limit_ns) || *abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t vals = smem_addr(smem + stage * C_::kStageBytes);  // MMA operand B (K-major)
        const uint32_t gath = vals + kValBytes;                           // MMA operand A (MN-major)
        const int64_t left = ncols - static_cast<int64_t>(s) * kKC;
        const int ksteps = left >= kKC ? 4 : static_cast<int>(left / 16);
        for (int kk = 0; kk < ksteps; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(vals + kk * 32, 16, 1024);
#pragma unroll
          for (int a = 0; a < NACC; ++a) {
            if (a < nacc) {
              const uint64_t adesc = smem_desc_sw128(gath + a * 2 * kChunkBytes + kk * 2048, kChunkBytes, 1024);
              umma_f16(tmem + a * kH, adesc, bdesc, idesc, (s > 0 || kk > 0) ? 1u : 0u);
            }
          }
        }
        umma_commit(empty0 + 8 * stage);
        if (++stage == Q) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        umma_commit(accum_bar);
      } else {
        atomicOr(p.status, kDevTimeout);
        *abort_flag = 1;
        umma_commit(drain_bar);
        mbar_wait(drain_bar, 0, 1000000ull);
        mbar_arrive(accum_bar);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int sp = warp & 3;  // TMEM sub-partition this warp may read
    const int row0 = task.window * kH;
    const bool to_ws = task.slot >= 0;
    float *ws = to_ws ? p.workspace + static_cast<int64_t>(task.slot) * kH * p.N : nullptr;
    bool have = nstages > 0;
    if (have) {
      if (!mbar_wait(accum_bar, 0, p.wait_limit_ns)) {
        atomicOr(p.status, kDevTimeout);
        *abort_flag = 1;
        have = false;
      } else if (*abort_flag) {
        have = false;
      }
      tc_fence_after_sync();
    }
    for (int a = 0; a < nacc; ++a) {
      const int n = n0 + a * 128 + sp * 32 + lane;
      uint32_t v[16];
      if (have) {
        tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(sp * 32) << 16) + a * kH, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0u;
      }
      if (n < p.N) {
#pragma unroll
        for (int i = 0; i < kH; ++i) {
          if (to_ws) {
            ws[static_cast<int64_t>(i) * p.N + n] = __uint_as_float(v[i]);
          } else if (row0 + i < p.M) {
            store_out<OUT_BF16>(p.C, static_cast<int64_t>(row0 + i) * p.N + n, __uint_as_float(v[i]));
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C_::kTmemCols);
  }
}

template <int NACC, int Q, bool IN_BF16, bool OUT_BF16>
cudaError_t launch_variant(const CUtensorMap &tmV, const CUtensorMap &tmB, const WcsrParams &p,
                           cudaStream_t stream) {
  using C_ = Cfg<NACC, Q>;
  auto kern = wcsr_spmm_kernel<NACC, Q, IN_BF16, OUT_BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(p.n_tasks, (p.N + C_::kBN - 1) / C_::kBN);
  kern<<<grid, kThreads, C_::kSmemBytes, stream>>>(tmV, tmB, p);
  return cudaGetLastError();
}

template <int NACC, int Q>
cudaError_t launch_dtypes(const CUtensorMap &tmV, const CUtensorMap &tmB, const WcsrParams &p, bool in_bf16,
                          bool out_bf16, cudaStream_t s) {
  if (in_bf16)
    return out_bf16 ? launch_variant<NACC, Q, true, true>(tmV, tmB, p, s)
                    : launch_variant<NACC, Q, true, false>(tmV, tmB, p, s);
  return out_bf16 ? launch_variant<NACC, Q, false, true>(tmV, tmB, p, s)
                  : launch_variant<NACC, Q, false, false>(tmV, tmB, p, s);
}

// One thread per 4 consecutive columns of one row of one split window;
// blockIdx.x names the split window, threads stride over its 16 x N partials.
template <bool OUT_BF16>
__global__ void __launch_bounds__(256) wcsr_reduce_kernel(const WcsrSplit *splits, const float *ws, void *C,
                                                          int32_t M, int32_t N) {
  const WcsrSplit sp = splits[blockIdx.x];
  const int64_t per = static_cast<int64_t>(kH) * N;
  for (int64_t e = (static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x) * 4; e < per;
       e += static_cast<int64_t>(gridDim.y) * blockDim.x * 4) {
    const int r = static_cast<int>(e / N);
    const int row = sp.window * kH + r;
    if (row >= M) break;  // rows only grow with e
    const float *src = ws + static_cast<int64_t>(sp.slot_begin) * per + e;
    float4 acc = *reinterpret_cast<const float4 *>(src);
    for (int s = 1; s < sp.n_slots; ++s) {
      const float4 v = *reinterpret_cast<const float4 *>(src + s * per);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int64_t off = static_cast<int64_t>(row) * N + (e - static_cast<int64_t>(r) * N);
    if constexpr (OUT_BF16) {
      __nv_bfloat16 *c = reinterpret_cast<__nv_bfloat16 *>(C) + off;
      c[0] = __float2bfloat16_rn(acc.x);
      c[1] = __float2bfloat16_rn(acc.y);
      c[2] = __float2bfloat16_rn(acc.z);
      c[3] = __float2bfloat16_rn(acc.w);
    } else {
      *reinterpret_cast<float4 *>(reinterpret_cast<float *>(C) + off) = acc;
    }
  }
}

}  // namespace

cudaError_t launch_wcsr(const CUtensorMap &tmV, const CUtensorMap &tmB, const WcsrParams &p, bool in_bf16,
                        bool out_bf16, cudaStream_t stream) {
  if (p.n_tasks == 0 || p.N == 0) return cudaSuccess;
  if (p.N <= 128) return launch_dtypes<1, 10>(tmV, tmB, p, in_bf16, out_bf16, stream);
  return launch_dtypes<2, 6>(tmV, tmB, p, in_bf16, out_bf16, stream);
}

cudaError_t launch_wcsr_reduce(const WcsrSplit *splits, int32_t n_splits, const float *workspace, void *C,
                               int32_t M, int32_t N, bool out_bf16, cudaStream_t stream) {
  if (n_splits == 0 || N == 0) return cudaSuccess;
  const int64_t per4 = (static_cast<int64_t>(kH) * N) / 4;  // N % 8 == 0
  const int64_t blocks = (per4 + 255) / 256;
  dim3 grid(n_splits, static_cast<unsigned>(blocks < 1024 ? blocks : 1024));
  if (out_bf16)
    wcsr_reduce_kernel<true><<<grid, 256, 0, stream>>>(splits, workspace, C, M, N);
  else
    wcsr_reduce_kernel<false><<<grid, 256, 0, stream>>>(splits, workspace, C, M, N);
  return cudaGetLastError();
}

}  // namespace spmm
