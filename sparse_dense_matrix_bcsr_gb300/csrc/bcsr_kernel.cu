// bcsr_kernel.cu -- BCSR SpMM for sm_103a: TMA loads, a producer warp feeding
// tcgen05.mma through a Q-stage mbarrier ring, fp32 accumulators in TMEM.
//
// Method: "AsyncSparse", Section III-C and Fig. 4 (warp-specialised
// producer/consumer pipeline over the stored blocks of one block row, full[Q]
// and empty[Q] barriers with phase bits, the first MMA overwriting the
// accumulator), Section III-B (each 64x64 block and its 64 rows of B are one
// 2-D TMA load each).  On sm_103a the consumer is a single thread issuing
// tcgen05.mma into TMEM, and the product is computed transposed:
//   C^T[n, r] = sum_k B[k, n] * blk[r, k]
// so the dense dimension N (128 columns per accumulator) is the MMA's M and
// runs over the 128 TMEM lanes, and the 64 rows of a block row are the MMA's
// N.  B tiles are MN-major MMA operands, blocks K-major ones.
//
// CTA = one block row x one tile of BN = 128*NACC columns of C; 6 warps:
//   warp 0      TMA producer (lane 0 issues; the warp shares index loads)
//   warp 1      TMEM allocator and MMA issuer (lane 0 issues)
//   warps 2..5  epilogue: TMEM -> registers -> C (warp w reads lanes of
//               sub-partition w % 4)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace spmm {
namespace {

constexpr int kBlk = 64;                      // block rows = block cols = K per block
constexpr int kBlkBytes = kBlk * kBlk * 2;    // one 64x64 16-bit block
constexpr int kChunkBytes = 64 * 64 * 2;      // 64 rows (k) x 64 columns (n) of B
constexpr int kThreads = 192;

template <int NACC, int Q>
struct Cfg {
  static constexpr int kBN = 128 * NACC;
  static constexpr int kChunks = 2 * NACC;
  static constexpr int kStageBytes = kBlkBytes + kChunks * kChunkBytes;
  static constexpr int kTmemCols = NACC == 1 ? 64 : 128;
  static constexpr int kBarBytes = 1024;
  static constexpr int kSmemBytes = Q * kStageBytes + kBarBytes + 1024;  // + alignment slack
};

template <bool OUT_BF16>
__device__ __forceinline__ void store_c(void *C, int64_t off, float v) {
  if constexpr (OUT_BF16)
    reinterpret_cast<__nv_bfloat16 *>(C)[off] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float *>(C)[off] = v;
}

template <int NACC, int Q, bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bcsr_spmm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const BcsrParams p) {
  using C_ = Cfg<NACC, Q>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Q * C_::kStageBytes);
  // bars[0..Q): full, bars[Q..2Q): empty, bars[2Q]: accumulator ready, bars[2Q+1]: drain
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * Q + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int br = blockIdx.x;
  const int n0 = blockIdx.y * C_::kBN;
  const int64_t jb = p.block_row_ptr[br];
  const int64_t je = p.block_row_ptr[br + 1];
  const int nblk = static_cast<int>(je - jb);
  const int nvalid = min(C_::kBN, p.N - n0);
  const int nch = min(C_::kChunks, (nvalid + 63) / 64);   // B chunks that hold valid columns
  const int nacc = min(NACC, (nvalid + 127) / 128);       // accumulators that hold valid columns

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
    tma_prefetch_desc(&tmA);
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
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t jbase = jb; jbase < je && ok; jbase += 32) {
      // The warp loads the next 32 block-column indices at once.
      const int64_t jl = jbase + lane;
      const int32_t my_col = jl < je ? p.block_col_idx[jl] : 0;
      const int cnt = (je - jbase) < 32 ? static_cast<int>(je - jbase) : 32;
      for (int t = 0; t < cnt; ++t) {
        const int32_t bcol = __shfl_sync(0xffffffffu, my_col, t);
        if (lane == 0) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns) || *abort_flag) {
            ok = false;
          } else {
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t st = smem_addr(smem + stage * C_::kStageBytes);
            mbar_arrive_expect_tx(fb, kBlkBytes + nch * kChunkBytes);
            tma_load_2d(st, &tmA, fb, 0, static_cast<int32_t>((jbase + t) * kBlk));
            for (int c = 0; c < nch; ++c)
              tma_load_2d(st + kBlkBytes + c * kChunkBytes, &tmB, fb, n0 + c * 64, bcol * kBlk);
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (++stage == Q) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      atomicOr(p.status, kDevTimeout);
      *abort_flag = 1;
      // Let the loads already in flight land before the CTA exits.
      const int64_t first = issued > Q ? issued - Q : 0;
      for (int64_t i = first; i < issued; ++i)
        mbar_wait(full0 + 8 * (i % Q), static_cast<uint32_t>((i / Q) & 1), 1000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nblk > 0) {
      constexpr uint32_t idesc = idesc_f16(IN_BF16, /*a_mn_major=*/true, /*b_mn_major=*/false, 128, 64);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = 0; t < nblk; ++t) {
        if (!mbar_wait(full0 + 8 * stage, phase, p.wait_limit_ns) || *abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_blk = smem_addr(smem + stage * C_::kStageBytes);  // A block: MMA operand B
        const uint32_t b_til = a_blk + kBlkBytes;                          // B tile:  MMA operand A
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(a_blk + kk * 32, 16, 1024);
#pragma unroll
          for (int a = 0; a < NACC; ++a) {
            if (a < nacc) {
              const uint64_t adesc = smem_desc_sw128(b_til + a * 2 * kChunkBytes + kk * 2048, kChunkBytes, 1024);
              umma_f16(tmem + a * 64, adesc, bdesc, idesc, (t > 0 || kk > 0) ? 1u : 0u);
            }
          }
        }
        umma_commit(empty0 + 8 * stage);  // frees the stage once these MMAs have read it
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
        mbar_arrive(accum_bar);  // release the epilogue
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int sp = warp & 3;  // TMEM sub-partition this warp may read
    const int row0 = br * kBlk;
    if (nblk == 0) {
      for (int a = 0; a < nacc; ++a) {
        const int n = n0 + a * 128 + sp * 32 + lane;
        if (n < p.N)
          for (int r = 0; r < kBlk && row0 + r < p.M; ++r)
            store_c<OUT_BF16>(p.C, static_cast<int64_t>(row0 + r) * p.ldc + n, 0.0f);
      }
    } else {
      const bool ok = mbar_wait(accum_bar, 0, p.wait_limit_ns);
      if (!ok) {
        atomicOr(p.status, kDevTimeout);
        *abort_flag = 1;
      } else if (!*abort_flag) {
        tc_fence_after_sync();
        for (int a = 0; a < nacc; ++a) {
          const int n = n0 + a * 128 + sp * 32 + lane;
          const bool nok = n < p.N;
#pragma unroll
          for (int cb = 0; cb < kBlk / 16; ++cb) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(sp * 32) << 16) + a * 64 + cb * 16, v);
            tmem_ld_wait();
            if (nok) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int r = row0 + cb * 16 + i;
                if (r < p.M) store_c<OUT_BF16>(p.C, static_cast<int64_t>(r) * p.ldc + n, __uint_as_float(v[i]));
              }
            }
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
cudaError_t launch_variant(const CUtensorMap &tmA, const CUtensorMap &tmB, const BcsrParams &p,
                           cudaStream_t stream) {
  using C_ = Cfg<NACC, Q>;
  auto kern = bcsr_spmm_kernel<NACC, Q, IN_BF16, OUT_BF16>;
  static bool attr_set = false;  // per instantiation; the attribute is per device function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(p.n_block_rows, (p.N + C_::kBN - 1) / C_::kBN);
  kern<<<grid, kThreads, C_::kSmemBytes, stream>>>(tmA, tmB, p);
  return cudaGetLastError();
}

template <int NACC, int Q>
cudaError_t launch_dtypes(const CUtensorMap &tmA, const CUtensorMap &tmB, const BcsrParams &p, bool in_bf16,
                          bool out_bf16, cudaStream_t s) {
  if (in_bf16)
    return out_bf16 ? launch_variant<NACC, Q, true, true>(tmA, tmB, p, s)
                    : launch_variant<NACC, Q, true, false>(tmA, tmB, p, s);
  return out_bf16 ? launch_variant<NACC, Q, false, true>(tmA, tmB, p, s)
                  : launch_variant<NACC, Q, false, false>(tmA, tmB, p, s);
}

}  // namespace

cudaError_t launch_bcsr(const CUtensorMap &tmA, const CUtensorMap &tmB, const BcsrParams &p, bool in_bf16,
                        bool out_bf16, cudaStream_t stream) {
  if (p.n_block_rows == 0 || p.N == 0) return cudaSuccess;
  // Tile width: 128 columns when N is small, else 256 (two accumulators
  // sharing each loaded block).
  if (p.N <= 128) return launch_dtypes<1, 6>(tmA, tmB, p, in_bf16, out_bf16, stream);
  return launch_dtypes<2, 4>(tmA, tmB, p, in_bf16, out_bf16, stream);
}

}  // namespace spmm
