// bcsr_kernel.cu -- BCSR SpMM for sm_103a: TMA loads, a producer warp feeding
// tcgen05.mma through a Q-stage mbarrier ring, fp32 accumulators in TMEM, and
// TMA stores of C.
//
// Method: "AsyncSparse", Section III-C and Fig. 4 (warp-specialised
// producer/consumer pipeline over the stored blocks of one block row, full[Q]
// and empty[Q] barriers with phase bits, the first MMA overwriting the
// accumulator), Section III-B (each 64x64 block and its 64 rows of B are
// 2-D TMA loads).  On sm_103a the consumer is a single thread issuing
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
//   warp 0      producer: reads the block-row pointers and block-column
//               indices, waits for a free stage, writes the stage's tile
//               record to shared memory and issues its TMA loads (lane 0)
//   warp 1      TMEM allocator and MMA issuer (lane 0 issues); it learns the
//               tile layout from the stage records, so it never waits on a
//               global load, and hands each finished accumulator to the
//               epilogue with a record of its own
//   warps 2..5  epilogue: TMEM -> registers -> a per-warp staging area in
//               shared memory -> one TMA store per 32-column box (warp w reads
//               the TMEM lanes of sub-partition w % 4, i.e. 32 columns of C)
// A block row without stored blocks still passes through the pipeline as
// one stage without loads, so its rows of C are written (zeros) by the same
// TMA stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace spmm {
namespace {

constexpr int kBlk = 64;                      // block rows = block cols = K per block
constexpr int kBlkBytes = kBlk * kBlk * 2;    // one 64x64 16-bit block
constexpr int kChunkBytes = 64 * 64 * 2;      // 64 rows (k) x 64 columns (n) of B
constexpr int kTmaWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kBoxCols = 32;                  // C columns of one TMA store box (one epilogue warp)

// Stage record flags (producer -> MMA) and accumulator record flags (MMA -> epilogue).
constexpr int32_t kRecFirst = 1;  // first stored block of its tile
constexpr int32_t kRecLast = 2;   // last stage of its tile
constexpr int32_t kRecEmpty = 4;  // block row without stored blocks: no loads, no MMA, C rows = 0
constexpr int32_t kRecEnd = 8;    // no more tiles

struct TileRec {
  int32_t br;     // block row
  int32_t nt;     // column tile
  int32_t flags;
  int32_t pad_;
};

template <int NACC, int Q, bool OUT_BF16>
struct Cfg {
  static constexpr int kBN = 128 * NACC;
  static constexpr int kChunks = 2 * NACC;
  static constexpr int kStageBytes = kBlkBytes + kChunks * kChunkBytes;
  static constexpr int kAccCols = 64 * NACC;               // TMEM columns of one accumulator set
  static constexpr int kTmemCols = NACC == 1 ? 128 : 256;  // two sets
  static constexpr int kOutBytes = OUT_BF16 ? 2 : 4;
  static constexpr int kBoxBytes = kBoxCols * kBlk * kOutBytes;   // 64 rows x 32 columns of C
  static constexpr int kWarpStaging = NACC * kBoxBytes;           // one box per accumulator
  static constexpr int kStagingBytes = kEpiWarps * kWarpStaging;
  static constexpr int kMiscBytes = 1024;                         // barriers, records, TMEM address
  static constexpr int kSmemBytes = Q * kStageBytes + kStagingBytes + kMiscBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert((2 * Q + 6) * 8 + (Q + 2) * 16 + 16 <= kMiscBytes, "barrier area");
};

// Tile t -> (block row, column tile).  Consecutive tile ids walk kGroupN
// column tiles of the same block row, so the CTAs running at one time touch
// about kGroupN column slices of B at once (they stay in L2) instead of one.
constexpr int kGroupN = 8;
__device__ __forceinline__ void tile_coords(int64_t t, int n_block_rows, int n_col_tiles, int &br, int &nt) {
  const int64_t span = static_cast<int64_t>(n_block_rows) * kGroupN;
  const int64_t g = t / span;
  const int64_t r = t - g * span;
  const int gsz = min(kGroupN, n_col_tiles - static_cast<int>(g) * kGroupN);
  br = static_cast<int>(r / gsz);
  nt = static_cast<int>(g) * kGroupN + static_cast<int>(r % gsz);
}

template <int NACC, int Q, bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bcsr_spmm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const BcsrParams p) {
  using C_ = Cfg<NACC, Q, OUT_BF16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *staging = smem + Q * C_::kStageBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(staging + C_::kStagingBytes);
  // bars: full[Q], empty[Q], acc_full[2], acc_empty[2], drain (+ one spare slot)
  TileRec *tile_rec = reinterpret_cast<TileRec *>(bars + 2 * Q + 6);               // [Q]
  volatile TileRec *acc_rec = reinterpret_cast<volatile TileRec *>(tile_rec + Q);  // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tile_rec + Q + 2);
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
      mbar_init(full0 + 8 * q, 1);   // the producer's arrive (with the TMA transaction bytes)
      mbar_init(empty0 + 8 * q, 1);  // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 2);  // the MMA thread's arrive (record) + its commit (MMAs done)
      mbar_init(acce0 + 8 * b, kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), C_::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    int64_t seq = 0;  // stages produced
    bool ok = true;
    // Waits (whole warp) until the current stage is free.
    auto claim = [&]() -> bool {
      const bool r = mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns);
      return __shfl_sync(0xffffffffu, r && !*abort_flag, 0);
    };
    auto advance = [&]() {
      ++seq;
      if (++stage == Q) {
        stage = 0;
        phase ^= 1u;
      }
    };
    // Block-row extent of the first tile; the next tile's is loaded while
    // this one's stages are issued.
    int br = 0, nt = 0;
    int64_t jb = 0, je = 0;
    if (static_cast<int64_t>(blockIdx.x) < n_tiles) {
      tile_coords(blockIdx.x, p.n_block_rows, n_col_tiles, br, nt);
      jb = p.block_row_ptr[br];
      je = p.block_row_ptr[br + 1];
    }
    for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      int br_n = 0, nt_n = 0;
      int64_t jb_n = 0, je_n = 0;
      const int64_t tn = t + gridDim.x;
      if (tn < n_tiles) {
        tile_coords(tn, p.n_block_rows, n_col_tiles, br_n, nt_n);
        jb_n = p.block_row_ptr[br_n];
        je_n = p.block_row_ptr[br_n + 1];
      }
      const int n0 = nt * C_::kBN;
      const int nch = min(C_::kChunks, (p.N - n0 + 63) / 64);
      if (jb == je) {
        ok = claim();
        if (!ok) break;
        if (lane == 0) {
          tile_rec[stage] = TileRec{br, nt, kRecFirst | kRecLast | kRecEmpty, 0};
          mbar_arrive(full0 + 8 * stage);  // releases the record
        }
        advance();
      }
      for (int64_t jbase = jb; jbase < je && ok; jbase += 32) {
        // The warp loads the next 32 block-column indices at once.
        const int64_t jl = jbase + lane;
        const int32_t my_col = jl < je ? p.block_col_idx[jl] : 0;
        const int cnt = (je - jbase) < 32 ? static_cast<int>(je - jbase) : 32;
        for (int i = 0; i < cnt; ++i) {
          const int32_t bcol = __shfl_sync(0xffffffffu, my_col, i);
          ok = claim();
          if (!ok) break;
          if (lane == 0) {
            const int64_t j = jbase + i;
            const int32_t flags = (j == jb ? kRecFirst : 0) | (j == je - 1 ? kRecLast : 0);
            tile_rec[stage] = TileRec{br, nt, flags, 0};
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t st = smem_addr(smem + stage * C_::kStageBytes);
            mbar_arrive_expect_tx(fb, kBlkBytes + nch * kChunkBytes);  // also releases the record
            tma_load_2d(st, &tmA, fb, 0, static_cast<int32_t>(j * kBlk));
            for (int c = 0; c < nch; ++c)
              tma_load_2d(st + kBlkBytes + c * kChunkBytes, &tmB, fb, n0 + c * 64, bcol * kBlk);
          }
          advance();
        }
      }
      br = br_n;
      nt = nt_n;
      jb = jb_n;
      je = je_n;
    }
    if (ok) {
      // end marker for the MMA thread
      ok = claim();
      if (ok && lane == 0) {
        tile_rec[stage] = TileRec{-1, -1, kRecEnd, 0};
        mbar_arrive(full0 + 8 * stage);
      }
    }
    if (!ok && lane == 0) {
      atomicOr(p.status, kDevTimeout);
      *abort_flag = 1;
      // Let the loads already in flight land before the CTA exits.
      const int64_t first = seq > Q ? seq - Q : 0;
      for (int64_t i = first; i < seq; ++i)
        mbar_wait(full0 + 8 * (i % Q), static_cast<uint32_t>((i / Q) & 1), 1000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp takes the waits (see mbar_wait_warp); lane 0 issues.
    constexpr uint32_t idesc = idesc_f16(IN_BF16, /*a_mn_major=*/true, /*b_mn_major=*/false, 128, 64);
    const bool leader = lane == 0;
    uint32_t stage = 0, phase = 0;
    uint32_t tcount = 0;  // tiles finished
    uint32_t buf = 0;
    bool ok = true;
    while (true) {
      ok = mbar_wait_warp(full0 + 8 * stage, phase, p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
      if (!ok) break;
      const TileRec rec = tile_rec[stage];
      if (rec.flags & (kRecFirst | kRecEnd)) {
        // Wait until the epilogue has drained this accumulator set.
        buf = tcount & 1u;
        const bool r = mbar_wait_warp(acce0 + 8 * buf, ((tcount >> 1) & 1u) ^ 1u, p.wait_limit_ns);
        ok = __shfl_sync(0xffffffffu, r && !*abort_flag, 0);
        if (!ok) break;
        tc_fence_after_sync();
      }
      if (rec.flags & kRecEnd) {
        if (leader) {
          acc_rec[buf].flags = kRecEnd;
          mbar_arrive(accf0 + 8 * buf);
          mbar_arrive(accf0 + 8 * buf);
        }
        break;
      }
      if (leader) {
        if (!(rec.flags & kRecEmpty)) {
          tc_fence_after_sync();
          const int nacc = min(NACC, (p.N - rec.nt * C_::kBN + 127) / 128);
          const uint32_t a_blk = smem_addr(smem + stage * C_::kStageBytes);  // A block: MMA operand B
          const uint32_t b_til = a_blk + kBlkBytes;                          // B tile:  MMA operand A
          const uint32_t acc = tmem + buf * C_::kAccCols;
          const bool first = (rec.flags & kRecFirst) != 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = smem_desc_sw128(a_blk + kk * 32, 16, 1024);
#pragma unroll
            for (int a = 0; a < NACC; ++a) {
              if (a < nacc) {
                const uint64_t adesc = smem_desc_sw128(b_til + a * 2 * kChunkBytes + kk * 2048, kChunkBytes, 1024);
                umma_f16(acc + a * 64, adesc, bdesc, idesc, (first && kk == 0) ? 0u : 1u);
              }
            }
          }
        }
        umma_commit(empty0 + 8 * stage);  // frees the stage once these MMAs have read it
        if (rec.flags & kRecLast) {
          acc_rec[buf].br = rec.br;
          acc_rec[buf].nt = rec.nt;
          acc_rec[buf].flags = rec.flags & kRecEmpty;
          mbar_arrive(accf0 + 8 * buf);  // releases the record
          umma_commit(accf0 + 8 * buf);  // arrives when the tile's MMAs are done
        }
      }
      if (rec.flags & kRecLast) ++tcount;
      __syncwarp();
      if (++stage == Q) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      if (leader) {
        atomicOr(p.status, kDevTimeout);
        *abort_flag = 1;
        umma_commit(drain_bar);
      }
      mbar_wait_warp(drain_bar, 0, 1000000ull);
      if (leader) {
        // let the epilogue see the abort flag without waiting out its limit
        for (int b = 0; b < 2; ++b) {
          mbar_arrive(accf0 + 8 * b);
          mbar_arrive(accf0 + 8 * b);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int sp = warp & 3;  // TMEM sub-partition this warp may read: C columns sp*32 .. sp*32+31 of each 128
    uint8_t *stg = staging + (warp - kEpiWarp0) * C_::kWarpStaging;
    const uint32_t stg_addr = smem_addr(stg);
    uint32_t tcount = 0;
    while (true) {
      const uint32_t buf = tcount & 1u;
      const bool r = mbar_wait_warp(accf0 + 8 * buf, (tcount >> 1) & 1u, p.wait_limit_ns);
      if (!__shfl_sync(0xffffffffu, r && !*abort_flag, 0)) {
        if (lane == 0 && !r) {
          atomicOr(p.status, kDevTimeout);
          *abort_flag = 1;
        }
        break;
      }
      const int32_t flags = acc_rec[buf].flags;
      if (flags & kRecEnd) break;
      const int br = acc_rec[buf].br;
      const int n0 = acc_rec[buf].nt * C_::kBN;
      const int nacc = min(NACC, (p.N - n0 + 127) / 128);
      tc_fence_after_sync();
      // the staging area is free once this warp's previous stores have read it
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      const uint32_t acc = tmem + buf * C_::kAccCols + (static_cast<uint32_t>(sp * 32) << 16);
      for (int a = 0; a < nacc; ++a) {
#pragma unroll
        for (int cb = 0; cb < kBlk / 16; ++cb) {
          uint32_t v[16];
          if (!(flags & kRecEmpty)) {
            tmem_ld_32x32b_x16(acc + a * 64 + cb * 16, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0u;
          }
          // row r of this warp's box: 32 consecutive columns, one per lane
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int r = cb * 16 + i;
            if constexpr (OUT_BF16)
              reinterpret_cast<__nv_bfloat16 *>(stg + a * C_::kBoxBytes)[r * kBoxCols + lane] =
                  __float2bfloat16_rn(__uint_as_float(v[i]));
            else
              reinterpret_cast<float *>(stg + a * C_::kBoxBytes)[r * kBoxCols + lane] = __uint_as_float(v[i]);
          }
        }
      }
      // This warp's reads of the accumulator set are complete.
      tc_fence_before_sync();
      fence_proxy_async_smem();  // the staging writes -> the TMA engine's reads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(acce0 + 8 * buf);
        for (int a = 0; a < nacc; ++a) {
          const int x = n0 + a * 128 + sp * 32;
          if (x < p.N) tma_store_2d(&tmC, stg_addr + a * C_::kBoxBytes, x, br * kBlk);
        }
        bulk_commit_group();
      }
      ++tcount;
    }
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C_::kTmemCols);
  }
}

template <int NACC, int Q, bool IN_BF16, bool OUT_BF16>
cudaError_t launch_variant(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                           const BcsrParams &p, cudaStream_t stream) {
  using C_ = Cfg<NACC, Q, OUT_BF16>;
  auto kern = bcsr_spmm_kernel<NACC, Q, IN_BF16, OUT_BF16>;
  static bool attr_set = false;  // per instantiation; the attribute is per device function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t tiles = static_cast<int64_t>(p.n_block_rows) * ((p.N + C_::kBN - 1) / C_::kBN);
  const int64_t grid = tiles < p.max_ctas ? tiles : p.max_ctas;
  kern<<<static_cast<unsigned>(grid), kThreads, C_::kSmemBytes, stream>>>(tmA, tmB, tmC, p);
  return cudaGetLastError();
}

template <int NACC, int Q>
cudaError_t launch_dtypes(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                          const BcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t s) {
  if (in_bf16)
    return out_bf16 ? launch_variant<NACC, Q, true, true>(tmA, tmB, tmC, p, s)
                    : launch_variant<NACC, Q, true, false>(tmA, tmB, tmC, p, s);
  return out_bf16 ? launch_variant<NACC, Q, false, true>(tmA, tmB, tmC, p, s)
                  : launch_variant<NACC, Q, false, false>(tmA, tmB, tmC, p, s);
}

}  // namespace

cudaError_t launch_bcsr(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const BcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t stream) {
  if (p.n_block_rows == 0 || p.N == 0) return cudaSuccess;
  // Tile width: 128 columns when N is small, else 256 (two accumulators
  // sharing each loaded block).
  if (p.N <= 128) return launch_dtypes<1, 6>(tmA, tmB, tmC, p, in_bf16, out_bf16, stream);
  return launch_dtypes<2, 4>(tmA, tmB, tmC, p, in_bf16, out_bf16, stream);
}

}  // namespace spmm
