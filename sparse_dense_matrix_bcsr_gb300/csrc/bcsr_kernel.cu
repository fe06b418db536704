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
// Work unit ("tile") = one block row x one tile of BN = 128*NACC columns of
// C.  The kernel is persistent: CTA c takes tiles c, c + G, c + 2G, ... (G =
// grid size); see tile_coords for the order.  Two TMEM accumulators
// alternate between tiles, so the epilogue of one tile overlaps the loads and
// MMAs of the next (the paper's non-persistent grid cannot overlap them when
// one CTA fills an SM).  6 warps:
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
constexpr int kLsuWarps = 4;                  // cp.async producer warps
constexpr int kTmaWarp = kLsuWarps;           // TMA producer warp
constexpr int kMmaWarp = kLsuWarps + 1;       // TMEM allocator and MMA issuer
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (kLsuWarps + 2 + kEpiWarps);

template <int NACC, int Q, int LSU_CH>
struct Cfg {
  static_assert(LSU_CH >= 0 && LSU_CH <= 2 * NACC, "LSU chunks are a subset of the tile's chunks");
  static constexpr int kTmaChunks = 2 * NACC - LSU_CH;   // B chunks loaded by TMA (the first ones)
  static constexpr int kBN = 128 * NACC;
  static constexpr int kChunks = 2 * NACC;
  static constexpr int kStageBytes = kBlkBytes + kChunks * kChunkBytes;
  static constexpr int kAccCols = 64 * NACC;               // TMEM columns of one accumulator set
  static constexpr int kTmemCols = NACC == 1 ? 128 : 256;  // two sets
  static constexpr int kSmemBytes = Q * kStageBytes + 1024 + 1024;  // + barriers + alignment slack
};

// Tile t -> (block row, column tile).  Consecutive tile ids walk kGroupN
// column tiles of the same block row, so the CTAs running at one time touch
// about kGroupN column slices of B at once (they stay in L2) instead of one
// (whose rows, N elements apart, fall on few L2 slices when N is a large
// power of two).
constexpr int kGroupN = 8;
__device__ __forceinline__ void tile_coords(int64_t t, int n_block_rows, int n_col_tiles, int &br, int &nt) {
  const int64_t span = static_cast<int64_t>(n_block_rows) * kGroupN;
  const int64_t g = t / span;
  const int64_t r = t - g * span;
  const int gsz = min(kGroupN, n_col_tiles - static_cast<int>(g) * kGroupN);
  br = static_cast<int>(r / gsz);
  nt = static_cast<int>(g) * kGroupN + static_cast<int>(r % gsz);
}

template <bool OUT_BF16>
__device__ __forceinline__ void store_c(void *C, int64_t off, float v) {
  if constexpr (OUT_BF16)
    reinterpret_cast<__nv_bfloat16 *>(C)[off] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float *>(C)[off] = v;
}

template <int NACC, int Q, int LSU_CH, bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bcsr_spmm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const BcsrParams p) {
  using C_ = Cfg<NACC, Q, LSU_CH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Q * C_::kStageBytes);
  // bars: full[Q], empty[Q], acc_full[2], acc_empty[2], drain
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * Q + 5);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_col_tiles = (p.N + C_::kBN - 1) / C_::kBN;
  const int64_t n_tiles = static_cast<int64_t>(p.n_block_rows) * n_col_tiles;

  const uint32_t full0 = smem_addr(&bars[0]);
  const uint32_t empty0 = smem_addr(&bars[Q]);
  const uint32_t accf0 = smem_addr(&bars[2 * Q]);
  const uint32_t acce0 = smem_addr(&bars[2 * Q + 2]);
  const uint32_t drain_bar = smem_addr(&bars[2 * Q + 4]);

  if (threadIdx.x == 0) {
    for (int q = 0; q < Q; ++q) {
      // the TMA arrive (with its transaction bytes) + one arrive per cp.async lane
      mbar_init(full0 + 8 * q, 1 + (LSU_CH > 0 ? 32 * kLsuWarps : 0));
      mbar_init(empty0 + 8 * q, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), C_::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < kLsuWarps) {
    // ------------------------------------------------------------ cp.async producers
    // The last LSU_CH 64-column chunks of each B tile: 64 rows x LSU_CH*8
    // 16-byte units, copied with the 128-byte swizzle written by hand.
    if constexpr (LSU_CH > 0) {
      constexpr int kUnitsRow = LSU_CH * 8;
      constexpr int kCopies = 64 * kUnitsRow / (32 * kLsuWarps);
      constexpr int kRowsPerPass = 32 * kLsuWarps / kUnitsRow;
      const int pt = threadIdx.x;
      const int v = pt % kUnitsRow;
      const int k0 = pt / kUnitsRow;
      const uint16_t *Bp = reinterpret_cast<const uint16_t *>(p.B);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        int br, nt;
        tile_coords(t, p.n_block_rows, n_col_tiles, br, nt);
        const int n = nt * C_::kBN + C_::kTmaChunks * 64 + v * 8;
        const bool n_live = n < p.N;
        const uint32_t u = static_cast<uint32_t>(v & 7);
        const uint32_t dst_col = kBlkBytes + (C_::kTmaChunks + (v >> 3)) * kChunkBytes;
        const int64_t jb = p.block_row_ptr[br];
        const int64_t je = p.block_row_ptr[br + 1];
        for (int64_t jbase = jb; jbase < je && ok; jbase += 32) {
          const int64_t jl = jbase + lane;
          const int32_t my_col = jl < je ? p.block_col_idx[jl] : 0;
          const int cnt = (je - jbase) < 32 ? static_cast<int>(je - jbase) : 32;
          for (int i = 0; i < cnt; ++i) {
            const int32_t bcol = __shfl_sync(0xffffffffu, my_col, i);
            if (lane == 0) ok = mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns) && !*abort_flag;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const uint32_t st = smem_addr(smem + stage * C_::kStageBytes);
            const int64_t krow0 = static_cast<int64_t>(bcol) * kBlk + k0;
            const uint16_t *src0 = Bp + krow0 * p.N + n;
#pragma unroll
            for (int q = 0; q < kCopies; ++q) {
              const int k = k0 + q * kRowsPerPass;
              const bool live = n_live && (krow0 + q * kRowsPerPass) < p.K;
              const uint32_t dst = st + dst_col + k * 128 + ((u ^ static_cast<uint32_t>(k & 7)) << 4);
              cp_async_16(dst, live ? static_cast<const void *>(src0 + static_cast<int64_t>(q) * kRowsPerPass * p.N)
                                    : static_cast<const void *>(Bp),
                          live ? 16u : 0u);
            }
            cp_async_arrive_noinc(full0 + 8 * stage);
            if (++stage == Q) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      cp_async_wait<0>();
      if (!ok && lane == 0) {
        atomicOr(p.status, kDevTimeout);
        *abort_flag = 1;
      }
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      int br, nt;
      tile_coords(t, p.n_block_rows, n_col_tiles, br, nt);
      const int n0 = nt * C_::kBN;
      const int nch = min(C_::kTmaChunks, max(0, (p.N - n0 + 63) / 64));
      const int64_t jb = p.block_row_ptr[br];
      const int64_t je = p.block_row_ptr[br + 1];
      for (int64_t jbase = jb; jbase < je && ok; jbase += 32) {
        // The warp loads the next 32 block-column indices at once.
        const int64_t jl = jbase + lane;
        const int32_t my_col = jl < je ? p.block_col_idx[jl] : 0;
        const int cnt = (je - jbase) < 32 ? static_cast<int>(je - jbase) : 32;
        for (int i = 0; i < cnt; ++i) {
          const int32_t bcol = __shfl_sync(0xffffffffu, my_col, i);
          // the whole warp takes the wait (see mbar_wait_warp); lane 0 issues
          ok = mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns);
          ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
          if (!ok) break;
          if (lane == 0) {
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t st = smem_addr(smem + stage * C_::kStageBytes);
            mbar_arrive_expect_tx(fb, kBlkBytes + nch * kChunkBytes);
            tma_load_2d(st, &tmA, fb, 0, static_cast<int32_t>((jbase + i) * kBlk));
            for (int c = 0; c < nch; ++c)
              tma_load_2d(st + kBlkBytes + c * kChunkBytes, &tmB, fb, n0 + c * 64, bcol * kBlk);
          }
          ++issued;
          if (++stage == Q) {
            stage = 0;
            phase ^= 1u;
          }
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
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp takes the waits (see mbar_wait_warp); lane 0 issues.
    {
      constexpr uint32_t idesc = idesc_f16(IN_BF16, /*a_mn_major=*/true, /*b_mn_major=*/false, 128, 64);
      const bool leader = lane == 0;
      uint32_t stage = 0, phase = 0;
      uint32_t tcount = 0;  // non-empty tiles processed
      bool ok = true;
      for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        int br, nt;
        tile_coords(t, p.n_block_rows, n_col_tiles, br, nt);
        const int n0 = nt * C_::kBN;
        const int nacc = min(NACC, (p.N - n0 + 127) / 128);
        const int nblk = static_cast<int>(p.block_row_ptr[br + 1] - p.block_row_ptr[br]);
        if (nblk == 0) continue;
        const uint32_t buf = tcount & 1u;
        const uint32_t use = tcount >> 1;
        // Wait until the epilogue has drained this accumulator set.
        ok = mbar_wait_warp(acce0 + 8 * buf, (use & 1u) ^ 1u, p.wait_limit_ns);
        ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t acc = tmem + buf * C_::kAccCols;
        for (int j = 0; j < nblk; ++j) {
          ok = mbar_wait_warp(full0 + 8 * stage, phase, p.wait_limit_ns);
          ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
          if (!ok) break;
          if (leader) {
            tc_fence_after_sync();
            if constexpr (LSU_CH > 0) fence_proxy_async_smem();  // cp.async writes -> async-proxy MMA reads
            const uint32_t a_blk = smem_addr(smem + stage * C_::kStageBytes);  // A block: MMA operand B
            const uint32_t b_til = a_blk + kBlkBytes;                          // B tile:  MMA operand A
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bdesc = smem_desc_sw128(a_blk + kk * 32, 16, 1024);
#pragma unroll
              for (int a = 0; a < NACC; ++a) {
                if (a < nacc) {
                  const uint64_t adesc =
                      smem_desc_sw128(b_til + a * 2 * kChunkBytes + kk * 2048, kChunkBytes, 1024);
                  umma_f16(acc + a * 64, adesc, bdesc, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                }
              }
            }
            umma_commit(empty0 + 8 * stage);  // frees the stage once these MMAs have read it
          }
          __syncwarp();
          if (++stage == Q) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (leader) umma_commit(accf0 + 8 * buf);  // accumulator set ready for the epilogue
        ++tcount;
      }
      if (!ok) {
        if (leader) {
          atomicOr(p.status, kDevTimeout);
          *abort_flag = 1;
          umma_commit(drain_bar);
        }
        mbar_wait_warp(drain_bar, 0, 1000000ull);
        if (leader) {
          // release the epilogue of the tile that will not complete
          mbar_arrive(accf0);
          mbar_arrive(accf0 + 8);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int sp = warp & 3;  // TMEM sub-partition this warp may read
    uint32_t tcount = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
      int br, nt;
      tile_coords(t, p.n_block_rows, n_col_tiles, br, nt);
      const int n0 = nt * C_::kBN;
      const int nacc = min(NACC, (p.N - n0 + 127) / 128);
      const int nblk = static_cast<int>(p.block_row_ptr[br + 1] - p.block_row_ptr[br]);
      const int row0 = br * kBlk;
      if (nblk == 0) {
        for (int a = 0; a < nacc; ++a) {
          const int n = n0 + a * 128 + sp * 32 + lane;
          if (n < p.N)
            for (int r = 0; r < kBlk && row0 + r < p.M; ++r)
              store_c<OUT_BF16>(p.C, static_cast<int64_t>(row0 + r) * p.ldc + n, 0.0f);
        }
        continue;
      }
      const uint32_t buf = tcount & 1u;
      const uint32_t use = tcount >> 1;
      if (!mbar_wait_warp(accf0 + 8 * buf, use & 1u, p.wait_limit_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kDevTimeout);
          *abort_flag = 1;
        }
        break;
      }
      if (*abort_flag) break;
      tc_fence_after_sync();
      const uint32_t acc = tmem + buf * C_::kAccCols + (static_cast<uint32_t>(sp * 32) << 16);
      for (int a = 0; a < nacc; ++a) {
        const int n = n0 + a * 128 + sp * 32 + lane;
        const bool nok = n < p.N;
#pragma unroll
        for (int cb = 0; cb < kBlk / 16; ++cb) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(acc + a * 64 + cb * 16, v);
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
      // This warp's reads of the accumulator set are complete.
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * buf);
      ++tcount;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C_::kTmemCols);
  }
}

template <int NACC, int Q, int LSU_CH, bool IN_BF16, bool OUT_BF16>
cudaError_t launch_variant(const CUtensorMap &tmA, const CUtensorMap &tmB, const BcsrParams &p,
                           cudaStream_t stream) {
  using C_ = Cfg<NACC, Q, LSU_CH>;
  auto kern = bcsr_spmm_kernel<NACC, Q, LSU_CH, IN_BF16, OUT_BF16>;
  static bool attr_set = false;  // per instantiation; the attribute is per device function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t tiles = static_cast<int64_t>(p.n_block_rows) * ((p.N + C_::kBN - 1) / C_::kBN);
  const int64_t grid = tiles < p.max_ctas ? tiles : p.max_ctas;
  kern<<<static_cast<unsigned>(grid), kThreads, C_::kSmemBytes, stream>>>(tmA, tmB, p);
  return cudaGetLastError();
}

template <int NACC, int Q, int LSU_CH>
cudaError_t launch_dtypes(const CUtensorMap &tmA, const CUtensorMap &tmB, const BcsrParams &p, bool in_bf16,
                          bool out_bf16, cudaStream_t s) {
  if (in_bf16)
    return out_bf16 ? launch_variant<NACC, Q, LSU_CH, true, true>(tmA, tmB, p, s)
                    : launch_variant<NACC, Q, LSU_CH, true, false>(tmA, tmB, p, s);
  return out_bf16 ? launch_variant<NACC, Q, LSU_CH, false, true>(tmA, tmB, p, s)
                  : launch_variant<NACC, Q, LSU_CH, false, false>(tmA, tmB, p, s);
}

}  // namespace

cudaError_t launch_bcsr(const CUtensorMap &tmA, const CUtensorMap &tmB, const BcsrParams &p, bool in_bf16,
                        bool out_bf16, cudaStream_t stream) {
  if (p.n_block_rows == 0 || p.N == 0) return cudaSuccess;
  // Tile width: 128 columns when N is small, else 256 (two accumulators
  // sharing each loaded block).
  if (p.N <= 128) return launch_dtypes<1, 6, 0>(tmA, tmB, p, in_bf16, out_bf16, stream);
  return launch_dtypes<2, 4, 0>(tmA, tmB, p, in_bf16, out_bf16, stream);
}

}  // namespace spmm
