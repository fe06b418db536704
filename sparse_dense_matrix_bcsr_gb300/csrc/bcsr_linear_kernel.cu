// bcsr_linear_kernel.cu -- BCSR SpMM in the layout of a linear layer:
//   Y = X * A^T,   Y[n][m] = sum_k X[n][k] * A[m][k]
// with A (M x K) in BCSR, X (N x K) and Y (N x M) row-major.  X is the
// paper's dense operand B = X^T stored column-major, the layout the BCSR
// kernel of "AsyncSparse" reads (Section III-B: a tile of B is contiguous in
// the column-major layout) and the one its drop-in replacement of a linear
// layer works in (Section IV-D, Table III: the gate projection of a 7B-class
// model, activations of 64K tokens).
//
// The operands of the MMA are swapped against bcsr_kernel.cu: 128 rows of X
// are the M operand and the 64 x 64 block is the N operand, both K-major as
// they lie in memory, so TMEM holds Y's own layout (lane = row n of X,
// columns = the block row's 64 output features) and the epilogue writes
// contiguous 128-byte pieces of Y's rows.  One stage is the block (8 KB) and a
// 256-row tile of X (one 32 KB TMA box); its MMAs are 4 k-steps x 2 halves of
// M = 128, N = 64, K = 16.
//
// Work unit ("tile") = one block row x 256 rows of X.  Persistent CTAs take
// tiles t, t + G, ... in the order of tile_coords (kGroupN tiles of X of the
// same block row in a row, so the CTAs running together read a few X slices,
// which stay in L2); two TMEM accumulators alternate between tiles; two CTAs
// per SM.  6 warps, as in bcsr_kernel.cu: a TMA producer, an MMA issuer and
// four epilogue warps (warp w reads TMEM lanes 32 (w % 4) .. + 31, rows of X).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace spmm {
namespace {

constexpr int kBlk = 64;
constexpr int kBlkBytes = kBlk * kBlk * 2;
constexpr int kTileN = 256;                    // rows of X per tile
constexpr int kXBytes = kTileN * kBlk * 2;     // one 256 x 64 box of X
constexpr int kStageBytes = kBlkBytes + kXBytes;
constexpr int kQ = 2;                          // stages per CTA
constexpr int kNbuf = 2;                       // TMEM accumulators per CTA
constexpr int kAccCols = 2 * kBlk;             // two halves of 128 rows x 64 columns
constexpr int kTmemCols = kNbuf * kAccCols;
constexpr int kThreads = 192;
constexpr int kTmaWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kEpiWarps = 4;
constexpr int kPartBytes = 32 * 128;           // one store box: 32 rows of Y x 128 bytes
constexpr int kStagingBytes = kEpiWarps * kPartBytes;  // one staging buffer per warp
constexpr int kMiscBytes = 1024;
constexpr int kSmemBytes = kQ * kStageBytes + kStagingBytes + kMiscBytes + 1024;
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(2 * kTmemCols <= 512, "TMEM of two CTAs");

constexpr int32_t kRecFirst = 1, kRecLast = 2, kRecEmpty = 4, kRecEnd = 8;
struct TileRec {
  int32_t br;
  int32_t nt;
  int32_t flags;
  int32_t pad_;
};

constexpr int kGroupN = 8;
__device__ __forceinline__ void tile_coords(int64_t t, int n_block_rows, int n_tiles_n, int &br, int &nt) {
  const int64_t span = static_cast<int64_t>(n_block_rows) * kGroupN;
  const int64_t g = t / span;
  const int64_t r = t - g * span;
  const int gsz = min(kGroupN, n_tiles_n - static_cast<int>(g) * kGroupN);
  br = static_cast<int>(r / gsz);
  nt = static_cast<int>(g) * kGroupN + static_cast<int>(r % gsz);
}

// Y's parts per tile and warp: 2 halves of 128 rows (the warp's 32 rows of
// each) x 64 output features, as 128-byte box rows: one box per half for bf16
// Y, two (32 features each) for fp32.
template <bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 2)
    bcsr_linear_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmY, const BcsrParams p) {
  constexpr int kOutBytes = OUT_BF16 ? 2 : 4;
  constexpr int kBoxCols = 128 / kOutBytes;      // features per box row
  constexpr int kParts = 2 * (kBlk / kBoxCols);  // store boxes per warp and tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *staging = smem + kQ * kStageBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(staging + kStagingBytes);
  // bars: full[kQ], empty[kQ], acc_full[kNbuf], acc_empty[kNbuf], drain
  TileRec *tile_rec = reinterpret_cast<TileRec *>(bars + 2 * kQ + 2 * kNbuf + 2);  // [kQ]
  volatile TileRec *acc_rec = reinterpret_cast<volatile TileRec *>(tile_rec + kQ);  // [kNbuf]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tile_rec + kQ + kNbuf);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles_n = (p.N + kTileN - 1) / kTileN;
  const int64_t n_tiles = static_cast<int64_t>(p.n_block_rows) * n_tiles_n;
  const uint32_t full0 = smem_addr(&bars[0]);
  const uint32_t empty0 = smem_addr(&bars[kQ]);
  const uint32_t accf0 = smem_addr(&bars[2 * kQ]);
  const uint32_t acce0 = smem_addr(&bars[2 * kQ + kNbuf]);
  const uint32_t drain_bar = smem_addr(&bars[2 * kQ + 2 * kNbuf]);

  if (threadIdx.x == 0) {
    for (int q = 0; q < kQ; ++q) {
      mbar_init(full0 + 8 * q, 1);
      mbar_init(empty0 + 8 * q, 1);
    }
    for (int b = 0; b < kNbuf; ++b) {
      mbar_init(accf0 + 8 * b, 2);
      mbar_init(acce0 + 8 * b, kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmY);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    int64_t seq = 0;
    bool ok = true;
    auto claim = [&]() -> bool {
      const bool r = mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns);
      return __shfl_sync(0xffffffffu, r && !*abort_flag, 0);
    };
    auto advance = [&]() {
      ++seq;
      if (++stage == kQ) {
        stage = 0;
        phase ^= 1u;
      }
    };
    for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      int br, nt;
      tile_coords(t, p.n_block_rows, n_tiles_n, br, nt);
      const int64_t jb = p.block_row_ptr[br], je = p.block_row_ptr[br + 1];
      if (jb == je) {
        ok = claim();
        if (!ok) break;
        if (lane == 0) {
          tile_rec[stage] = TileRec{br, nt, kRecFirst | kRecLast | kRecEmpty, 0};
          mbar_arrive(full0 + 8 * stage);
        }
        advance();
      }
      for (int64_t jbase = jb; jbase < je && ok; jbase += 32) {
        const int64_t jl = jbase + lane;
        const int32_t my_col = jl < je ? p.block_col_idx[jl] : 0;
        const int cnt = (je - jbase) < 32 ? static_cast<int>(je - jbase) : 32;
        for (int i = 0; i < cnt; ++i) {
          const int32_t bcol = __shfl_sync(0xffffffffu, my_col, i);
          ok = claim();
          if (!ok) break;
          if (lane == 0) {
            const int64_t j = jbase + i;
            tile_rec[stage] = TileRec{br, nt, (j == jb ? kRecFirst : 0) | (j == je - 1 ? kRecLast : 0), 0};
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t st = smem_addr(smem + stage * kStageBytes);
            mbar_arrive_expect_tx(fb, kStageBytes);
            tma_load_2d(st, &tmA, fb, 0, static_cast<int32_t>(j * kBlk));
            tma_load_2d(st + kBlkBytes, &tmX, fb, bcol * kBlk, nt * kTileN);
          }
          advance();
        }
      }
    }
    if (ok) {
      ok = claim();
      if (ok && lane == 0) {
        tile_rec[stage] = TileRec{-1, -1, kRecEnd, 0};
        mbar_arrive(full0 + 8 * stage);
      }
    }
    if (!ok && lane == 0) {
      atomicOr(p.status, kDevTimeout);
      *abort_flag = 1;
      const int64_t first = seq > kQ ? seq - kQ : 0;
      for (int64_t i = first; i < seq; ++i)
        mbar_wait(full0 + 8 * (i % kQ), static_cast<uint32_t>((i / kQ) & 1), 1000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_f16(IN_BF16, /*a_mn_major=*/false, /*b_mn_major=*/false, 128, kBlk);
    const bool leader = lane == 0;
    uint32_t stage = 0, phase = 0, tcount = 0, buf = 0;
    bool ok = true;
    while (true) {
      ok = mbar_wait_warp(full0 + 8 * stage, phase, p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
      if (!ok) break;
      const TileRec rec = tile_rec[stage];
      if (rec.flags & (kRecFirst | kRecEnd)) {
        buf = tcount % kNbuf;
        const bool r = mbar_wait_warp(acce0 + 8 * buf, ((tcount / kNbuf) & 1u) ^ 1u, p.wait_limit_ns);
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
          const uint32_t blk = smem_addr(smem + stage * kStageBytes);  // N operand: 64 rows of A x 64 k
          const uint32_t xt = blk + kBlkBytes;                         // M operand: 256 rows of X x 64 k
          const uint32_t acc = tmem + buf * kAccCols;
          const bool first = (rec.flags & kRecFirst) != 0;
          // half h: rows 128h .. 128h + 127 of the tile
          const uint64_t bdesc0 = smem_desc_sw128(blk, 16, 1024);
          const uint64_t adesc0 = smem_desc_sw128(xt, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = smem_desc_add(bdesc0, kk * 32);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              umma_f16(acc + h * kBlk, smem_desc_add(adesc0, h * (kXBytes / 2) + kk * 32), bdesc, idesc,
                       (first && kk == 0) ? 0u : 1u);
          }
        }
        umma_commit(empty0 + 8 * stage);
        if (rec.flags & kRecLast) {
          acc_rec[buf].br = rec.br;
          acc_rec[buf].nt = rec.nt;
          acc_rec[buf].flags = rec.flags & kRecEmpty;
          mbar_arrive(accf0 + 8 * buf);
          umma_commit(accf0 + 8 * buf);
        }
      }
      if (rec.flags & kRecLast) ++tcount;
      __syncwarp();
      if (++stage == kQ) {
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
      if (leader)
        for (int b = 0; b < kNbuf; ++b) {
          mbar_arrive(accf0 + 8 * b);
          mbar_arrive(accf0 + 8 * b);
        }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w holds rows 32 (w % 4) + lane of each 128-row half (TMEM lanes)
    // and the block row's 64 features (TMEM columns h * 64 ..).  Each part
    // (one store box: 32 rows x 128 bytes) goes through the warp's staging
    // buffer in the 128-byte swizzled layout of the store, reused once the
    // previous store has read it.
    const int sp = warp & 3;
    uint8_t *stg = staging + (warp - kEpiWarp0) * kPartBytes;
    const uint32_t row_sw = static_cast<uint32_t>(lane & 7);
    uint32_t tcount = 0;
    while (true) {
      const uint32_t buf = tcount % kNbuf;
      const bool r = mbar_wait_warp(accf0 + 8 * buf, (tcount / kNbuf) & 1u, p.wait_limit_ns);
      if (!__shfl_sync(0xffffffffu, r && !*abort_flag, 0)) {
        if (lane == 0 && !r) {
          atomicOr(p.status, kDevTimeout);
          *abort_flag = 1;
        }
        break;
      }
      const int32_t flags = acc_rec[buf].flags;
      if (flags & kRecEnd) break;
      const bool zero = (flags & kRecEmpty) != 0;
      const int m0 = acc_rec[buf].br * kBlk;
      const int n0 = acc_rec[buf].nt * kTileN + sp * 32;
      tc_fence_after_sync();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(sp * 32) << 16) + buf * kAccCols;
#pragma unroll 1
      for (int part = 0; part < kParts; ++part) {
        const int h = part / (kParts / 2);             // half of the tile
        const int c0 = (part % (kParts / 2)) * kBoxCols;  // first feature of the part
        uint8_t *pst = stg;
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        // kBoxCols features = kBoxCols / 16 TMEM loads of 16 columns
        uint32_t v[kBoxCols / 16][16];
#pragma unroll
        for (int g = 0; g < kBoxCols / 16; ++g) {
          if (!zero) {
            tmem_ld_32x32b_x16(tbase + h * kBlk + c0 + g * 16, v[g]);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[g][i] = 0u;
          }
        }
        if (!zero) tmem_ld_wait();
        uint8_t *row = pst + lane * 128;
#pragma unroll
        for (int g = 0; g < kBoxCols / 16; ++g) {
          if constexpr (OUT_BF16) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const __nv_bfloat162 b2 =
                  __floats2bfloat162_rn(__uint_as_float(v[g][2 * i]), __uint_as_float(v[g][2 * i + 1]));
              w[i] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            const uint32_t u0 = static_cast<uint32_t>(g * 2);
            *reinterpret_cast<uint4 *>(row + (((u0 + 0) ^ row_sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4 *>(row + (((u0 + 1) ^ row_sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
          } else {
            const uint32_t u0 = static_cast<uint32_t>(g * 4);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4 *>(row + (((u0 + q) ^ row_sw) << 4)) =
                  make_uint4(v[g][4 * q], v[g][4 * q + 1], v[g][4 * q + 2], v[g][4 * q + 3]);
          }
        }
        if (part == kParts - 1) tc_fence_before_sync();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (part == kParts - 1) mbar_arrive(acce0 + 8 * buf);
          const int y = n0 + h * 128;
          if (y < p.N && m0 + c0 < p.M) tma_store_2d(&tmY, smem_addr(pst), m0 + c0, y);
          bulk_commit_group();
        }
      }
      ++tcount;
    }
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool IN_BF16, bool OUT_BF16>
cudaError_t launch_linear_variant(const CUtensorMap &tmA, const CUtensorMap &tmX, const CUtensorMap &tmY,
                                  const BcsrParams &p, cudaStream_t stream) {
  auto kern = bcsr_linear_kernel<IN_BF16, OUT_BF16>;
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_smem_limit_once(kern, kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const int64_t tiles = static_cast<int64_t>(p.n_block_rows) * ((p.N + kTileN - 1) / kTileN);
  const int64_t cap = p.max_ctas > 0 ? p.max_ctas : 2ll * p.num_sms;
  const int64_t grid = tiles < cap ? tiles : cap;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tmA, tmX, tmY, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bcsr_linear(const CUtensorMap &tmA, const CUtensorMap &tmX, const CUtensorMap &tmY,
                               const BcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t stream) {
  if (p.n_block_rows == 0 || p.N == 0) return cudaSuccess;
  if (in_bf16)
    return out_bf16 ? launch_linear_variant<true, true>(tmA, tmX, tmY, p, stream)
                    : launch_linear_variant<true, false>(tmA, tmX, tmY, p, stream);
  return out_bf16 ? launch_linear_variant<false, true>(tmA, tmX, tmY, p, stream)
                  : launch_linear_variant<false, false>(tmA, tmX, tmY, p, stream);
}

}  // namespace spmm
