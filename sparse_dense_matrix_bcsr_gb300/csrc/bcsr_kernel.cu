// bcsr_kernel.cu -- BCSR SpMM for sm_103a: TMA loads, a producer warp feeding
// tcgen05.mma through a Q-stage mbarrier ring, fp32 accumulators in TMEM, and
// TMA stores of C.
//
// Method: "AsyncSparse", Section III-C and Fig. 4 (warp-specialised
// producer/consumer pipeline over the stored blocks of one block row, full[Q]
// and empty[Q] barriers with phase bits, the first MMA overwriting the
// accumulator), Section III-B (each 64x64 block and its 64 rows of B are
// 2-D TMA loads).  On sm_103a the consumer is one warp issuing
// tcgen05.mma into TMEM:
//   C[r, n] += sum_k blk[r, k] * B[k, n]
// with the block as the M = 64 operand (K-major) and the B tile as the N
// operand (MN-major).  On GB300 an M=128 x N=64 MMA costs as long as an
// M=64 x N=128 one (about 97 cycles), and the weight-stationary M=64 x N=256
// form takes about 93 cycles for four times the work, so the block rows are
// the MMA's M and the dense columns its N (see Cfg for the TMEM layouts).
//
// Work unit ("tile") = one block row x BN columns of C.  The kernel is
// persistent: CTA c takes tiles c, c + G, c + 2G, ... (G = grid size); see
// tile_coords for the order.  Two TMEM accumulators alternate between tiles,
// so the epilogue of one tile overlaps the loads and MMAs of the next (with a
// single accumulator the tensor pipe drains at every tile boundary: 13%
// slower on GB300).  Wide tiles run two CTAs per SM when there are enough.
// 6 warps:
//   warp 0      producer: reads the block-row pointers and block-column
//               indices, waits for a free stage, writes the stage's tile
//               record to shared memory and issues its TMA loads (lane 0)
//   warp 1      TMEM allocator and MMA issuer (converged; one elected lane
//               issues each MMA and commit); it learns the
//               tile layout from the stage records, so it never waits on a
//               global load, and hands each finished accumulator to the
//               epilogue with a record of its own
//   warps 2..5  epilogue: TMEM -> registers -> a per-warp staging area in
//               shared memory -> TMA stores (warp w reads the TMEM lanes of
//               sub-partition w % 4; which rows and columns those hold
//               depends on the tile width, see Cfg)
// A block row without stored blocks still passes through the pipeline as
// one stage without loads, so its rows of C are written (zeros) by the same
// TMA stores.
//
// Split schedule (BcsrParams::split_grid > 0), for problems with too few
// tiles to keep every SM busy (the paper's static grid of one CTA per tile,
// Section III-F, leaves SMs idle there): the stages of all tiles are listed
// tile after tile, and CTA c takes an equal contiguous share of that list, so
// a tile's blocks may be spread over several CTAs.  A CTA's run of stages of
// one tile is a "segment"; a segment holding the whole tile is stored to C as
// usual, a cut one is written as fp32 partial sums to the CTA's workspace
// slot and split_reduce_kernel adds the slots of each cut tile in CTA order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "split_reduce.cuh"

namespace spmm {
namespace {

constexpr int kBlk = 64;                      // block rows = block cols = K per block
constexpr int kBlkBytes = kBlk * kBlk * 2;    // one 64x64 16-bit block
constexpr int kChunkBytes = 64 * 64 * 2;      // 64 rows (k) x 64 columns (n) of B
constexpr int kEpiWarps = 4;
constexpr int kBoxBytes = 2048;               // one TMA store box of C in shared memory

// Stage record flags (producer -> MMA) and accumulator record flags (MMA -> epilogue).
constexpr int32_t kRecFirst = 1;       // first stage of a segment: the MMA overwrites the accumulator
constexpr int32_t kRecLast = 2;        // last stage of a segment: the accumulator goes to the epilogue
constexpr int32_t kRecEmpty = 4;       // block row without stored blocks: no loads, no MMA, C rows = 0
constexpr int32_t kRecEnd = 8;         // no more tiles
constexpr int32_t kRecTileFirst = 16;  // the tile's first stage
constexpr int32_t kRecTileLast = 32;   // the tile's last stage
constexpr int32_t kRecAtF0 = 64;       // the CTA's first stage (split schedule: partial slot 2c, else 2c + 1)
constexpr int32_t kRecWhole = kRecTileFirst | kRecTileLast;

struct TileRec {
  int32_t br;     // block row
  int32_t nt;     // column tile
  int32_t flags;
  int32_t nblk;   // blocks in the stage (1 .. KB)
};

// BN columns per tile, Q pipeline stages, NBUF TMEM accumulators, the
// epilogue writing each warp's share of a tile in PARTS column parts through
// two alternating staging buffers, MINB CTAs per SM, PW producer warps (warp
// w issues the stages s with s % PW == w; warps PW and PW+1..PW+4 are the MMA
// issuer and the epilogue), KB consecutive blocks of a block row per stage
// (each with its own B tile; more MMA work per barrier handshake, whose fixed
// cost bounds problems with few long block rows).
//
// Narrow tiles (BN = 128) use the plain MMA, M = 64 x N = 128: the
// accumulator's rows 16s..16s+15 sit in TMEM lanes 32s..32s+15, so epilogue
// warp s holds 16 rows x BN columns and stores 16-row x 128-byte boxes (128-byte
// swizzle).  Wide tiles (BN = 256) use the weight-stationary MMA, M = 64 x
// N = 256 (~93 cycles on GB300 against 128): rows 0..63 sit in lanes 0..63 for
// columns 0..127 and in lanes 64..127 for columns 128..255, in 128 TMEM
// columns, so warp s holds rows 32(s%2)..32(s%2)+31 x columns 128(s/2) ..
// 128(s/2)+127 and stores 32-row x 64-byte boxes (64-byte swizzle).
template <int BN, int Q, int NBUF, int PARTS, int MINB, int PW, int KB, bool OUT_BF16>
struct Cfg {
  static constexpr int kMmaWarp = PW;
  static constexpr int kEpiWarp0 = PW + 1;
  static constexpr int kThreads = 32 * (PW + 1 + kEpiWarps);
  static constexpr int kBN = BN;
  static constexpr bool kWS = BN >= 256;                      // weight-stationary MMA
  static constexpr int kNmma = BN < 256 ? BN : 256;           // N of one MMA
  static constexpr int kMmas = BN / kNmma;                    // MMAs per 16-deep k step
  static constexpr int kChunks = BN / 64;                     // 64-column chunks of the B tile
  static constexpr int kSubBytes = kBlkBytes + kChunks * kChunkBytes;   // one block and its B tile
  static constexpr int kStageBytes = KB * kSubBytes;
  static constexpr int kAccCols = kWS ? BN / 2 : BN;          // TMEM columns of one accumulator
  static constexpr int kTmemCols = NBUF * kAccCols;
  static constexpr int kOutBytes = OUT_BF16 ? 2 : 4;
  static constexpr int kWarpRows = kWS ? 32 : 16;             // rows of C an epilogue warp holds
  static constexpr int kWarpCols = kWS ? BN / 2 : BN;         // columns of C an epilogue warp holds
  static constexpr int kRowBytes = kWS ? 64 : 128;            // bytes of a store box row
  static constexpr int kBoxCols = kRowBytes / kOutBytes;      // C columns of one store box
  static constexpr int kPartCols = kWarpCols / PARTS;
  static constexpr int kPartGroups = kPartCols / 16;          // 16-column TMEM loads per part
  static constexpr int kBatch = kPartGroups < 4 ? kPartGroups : 4;  // TMEM loads per wait
  static constexpr int kBatches = kPartGroups / kBatch;
  static constexpr int kPartBoxes = kPartCols / kBoxCols;     // store boxes per part
  static constexpr int kPartBytes = kPartBoxes * kBoxBytes;
  static constexpr int kWarpStaging = 2 * kPartBytes;
  static constexpr int kStagingBytes = kEpiWarps * kWarpStaging;
  static constexpr int kMiscBytes = 1024;                     // barriers, records, TMEM address
  static constexpr int kSmemBytes = Q * kStageBytes + kStagingBytes + kMiscBytes + 1024;  // + alignment slack
  static_assert(kWarpRows * kRowBytes == kBoxBytes, "store box");
  static_assert(kSmemBytes <= 227 * 1024 && MINB * (kSmemBytes + 1024) <= 228 * 1024, "shared memory");
  static_assert(MINB * kTmemCols <= 512 && (kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512), "TMEM");
  static_assert((2 * Q + 6) * 8 + (Q + 2) * 16 + 16 <= kMiscBytes, "barrier area");
  // A producer warp waits on a stage's empty barrier once per use of that
  // stage it owns; with PW <= Q the phase it waits for is never two phases
  // ahead of the barrier, so the parity test cannot pass early.
  static_assert(PW >= 1 && PW <= Q, "producer warps");
  static_assert(KB == 1 || KB == 2, "blocks per stage");
  static_assert(BN % 128 == 0 && BN <= 256 && kNmma % 16 == 0 && kPartBoxes >= 1 && PARTS % 2 == 0 &&
                    kPartGroups % kBatch == 0, "tile shape");
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

template <int BN, int Q, int NBUF, int PARTS, int MINB, int PW, int KB, bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(Cfg<BN, Q, NBUF, PARTS, MINB, PW, KB, OUT_BF16>::kThreads, MINB)
    bcsr_spmm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const BcsrParams p) {
  using C_ = Cfg<BN, Q, NBUF, PARTS, MINB, PW, KB, OUT_BF16>;
  constexpr int kMmaWarp = C_::kMmaWarp;
  constexpr int kEpiWarp0 = C_::kEpiWarp0;
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
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(accf0 + 8 * b, 2);  // the MMA thread's arrive (record) + its commit (MMAs done)
      mbar_init(acce0 + 8 * b, kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    if (p.split_grid > 0) {  // this CTA's partial-sum records (overwritten below when used)
      p.partials[2 * blockIdx.x] = PartialRec{-1, 0, 0, 0};
      p.partials[2 * blockIdx.x + 1] = PartialRec{-1, 0, 0, 0};
    }
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

  if (warp < PW) {
    // ------------------------------------------------------------ producer
    // Every producer warp walks the same stage sequence; warp pw claims and
    // issues the stages s with s % PW == pw and only counts the others.
    const int pw = warp;
    uint32_t stage = 0, phase = 0;
    int64_t seq = 0;  // stages produced
    bool ok = true;
    auto mine = [&]() { return PW == 1 || static_cast<int>(seq % PW) == pw; };
    // Waits (whole warp) until the current stage is free, if it is this warp's.
    auto claim = [&]() -> bool {
      if (!mine()) return true;
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
    // One stage: its tile record (released to the MMA thread by the arrive)
    // and, unless the block row is empty, the TMA loads of blocks j .. j+nblk-1
    // and of the 64 rows of B each multiplies (block columns bcol0, bcol1) for
    // column tile nt.
    auto issue = [&](int br, int nt, int64_t j, int32_t bcol0, int32_t bcol1, int nblk, int32_t flags) {
      if (lane == 0 && mine()) {
        tile_rec[stage] = TileRec{br, nt, flags, nblk};
        const uint32_t fb = full0 + 8 * stage;
        if (flags & kRecEmpty) {
          mbar_arrive(fb);
        } else {
          const int n0 = nt * C_::kBN;
          const int nch = min(C_::kChunks, (p.N - n0 + 63) / 64);
          const uint32_t st = smem_addr(smem + stage * C_::kStageBytes);
          mbar_arrive_expect_tx(fb, nblk * (kBlkBytes + nch * kChunkBytes));
          for (int b = 0; b < nblk; ++b) {
            const uint32_t sb = st + b * C_::kSubBytes;
            tma_load_2d(sb, &tmA, fb, 0, static_cast<int32_t>((j + b) * kBlk));
            for (int c = 0; c < nch; ++c)
              tma_load_2d(sb + kBlkBytes + c * kChunkBytes, &tmB, fb, n0 + c * 64, (b ? bcol1 : bcol0) * kBlk);
          }
        }
      }
      advance();
    };
    if (p.split_grid > 0) {
      // Split schedule: stages of all tiles in tile order (tile_coords), a
      // tile's stages being its block row's blocks in order (one empty stage
      // for a block row without blocks); this CTA takes [f0, f1).  Within a
      // group of kGroupN column tiles, tile (br, i) starts at stage
      // gsz * P[br] + i * len(br) of the group, P = stage_row_ptr.
      const int nbr = p.n_block_rows;
      const int64_t s_all = p.split_stages;  // stages per column tile (= P[nbr])
      const int64_t total = s_all * n_col_tiles;
      const int64_t f0 = total * blockIdx.x / gridDim.x;
      const int64_t f1 = total * (blockIdx.x + 1) / gridDim.x;
      const int64_t n_blocks = p.n_blocks;
      const int64_t span = s_all * kGroupN;
      int g = static_cast<int>(f0 / span);
      int64_t r = f0 - g * span;
      int gsz = min(kGroupN, n_col_tiles - g * kGroupN);
      // Last block row with gsz * P[br] <= r, found 32 samples of P at a time
      // by the whole warp (the range shrinks 32-fold per round of loads).
      int lo = 0, hi = nbr - 1;
      while (hi > lo) {
        const int64_t span_r = hi - lo;
        const int idx = lo + static_cast<int>((span_r * (lane + 1) + 31) / 32);  // in (lo, hi], lane 31: hi
        const unsigned ok = __ballot_sync(0xffffffffu, gsz * p.stage_row_ptr[idx] <= r);
        if (ok == 0) {
          hi = __shfl_sync(0xffffffffu, idx, 0) - 1;
        } else {
          const int k = 31 - __clz(static_cast<int>(ok));
          const int idx_k = __shfl_sync(0xffffffffu, idx, k);
          const int idx_n = __shfl_sync(0xffffffffu, idx, k < 31 ? k + 1 : 31);
          hi = k < 31 ? idx_n - 1 : hi;
          lo = idx_k;
        }
      }
      int br = lo;
      int64_t len = p.stage_row_ptr[br + 1] - p.stage_row_ptr[br];
      r -= gsz * p.stage_row_ptr[br];
      int i = static_cast<int>(r / len);
      int64_t j = r - i * len;  // stage within the tile
      int64_t jb = p.block_row_ptr[br], je = p.block_row_ptr[br + 1];
      // the warp holds 32 consecutive block-column indices from `cbase`
      int64_t cbase = -64;
      int32_t cval = 0;
      for (int64_t f = f0; f < f1; ++f) {
        const bool empty = je == jb;
        int32_t bcol = 0;
        if (!empty) {
          const int64_t x = jb + j;
          if (x < cbase || x >= cbase + 32) {
            cbase = x;
            cval = x + lane < n_blocks ? p.block_col_idx[x + lane] : 0;
          }
          bcol = __shfl_sync(0xffffffffu, cval, static_cast<int>(x - cbase));
        }
        ok = claim();
        if (!ok) break;
        const bool tfirst = j == 0, tlast = j == len - 1;
        const int32_t flags = (tfirst || f == f0 ? kRecFirst : 0) | (tlast || f == f1 - 1 ? kRecLast : 0) |
                              (tfirst ? kRecTileFirst : 0) | (tlast ? kRecTileLast : 0) | (f == f0 ? kRecAtF0 : 0) |
                              (empty ? kRecEmpty : 0);
        issue(br, g * kGroupN + i, jb + j, bcol, 0, 1, flags);
        if (++j == len) {  // next tile
          j = 0;
          if (++i == gsz) {
            i = 0;
            if (++br == nbr) {
              br = 0;
              ++g;
              gsz = min(kGroupN, n_col_tiles - g * kGroupN);
            }
            if (f + 1 < f1) {
              jb = p.block_row_ptr[br];
              je = p.block_row_ptr[br + 1];
              len = p.stage_row_ptr[br + 1] - p.stage_row_ptr[br];
            }
          }
        }
      }
    } else {
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
        if (jb == je) {
          ok = claim();
          if (!ok) break;
          issue(br, nt, 0, 0, 0, 1, kRecFirst | kRecLast | kRecWhole | kRecEmpty);
        }
        for (int64_t jbase = jb; jbase < je && ok; jbase += 32) {
          // The warp loads the next 32 block-column indices at once.
          const int64_t jl = jbase + lane;
          const int32_t my_col = jl < je ? p.block_col_idx[jl] : 0;
          const int cnt = (je - jbase) < 32 ? static_cast<int>(je - jbase) : 32;
          for (int i = 0; i < cnt; i += KB) {  // KB divides 32: a stage never spans two loads
            const int32_t bcol0 = __shfl_sync(0xffffffffu, my_col, i);
            const int32_t bcol1 = __shfl_sync(0xffffffffu, my_col, (i + 1) & 31);
            const int nb = min(KB, cnt - i);
            ok = claim();
            if (!ok) break;
            const int64_t j = jbase + i;
            issue(br, nt, j, bcol0, bcol1, nb,
                  (j == jb ? kRecFirst | kRecTileFirst : 0) | (j + nb - 1 == je - 1 ? kRecLast | kRecTileLast : 0));
          }
        }
        br = br_n;
        nt = nt_n;
        jb = jb_n;
        je = je_n;
      }
    }
    if (ok) {
      // end marker for the MMA thread
      ok = claim();
      if (ok && lane == 0 && mine()) {
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
        if (PW == 1 || static_cast<int>(i % PW) == pw)
          mbar_wait(full0 + 8 * (i % Q), static_cast<uint32_t>((i / Q) & 1), 1000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp takes the waits (see mbar_wait_warp) and issues
    // converged (one elected lane per MMA and commit); lane 0 writes records.
    constexpr uint32_t idesc = idesc_f16(IN_BF16, /*a_mn_major=*/false, /*b_mn_major=*/true, 64, C_::kNmma);
    const bool leader = lane == 0;
    uint32_t stage = 0, phase = 0;
    uint32_t tcount = 0;  // tiles finished
    uint32_t buf = 0;
    int32_t seg_flags = 0;  // kRecTileFirst / kRecAtF0 of the current segment's first stage
    bool ok = true;
    while (true) {
      ok = mbar_wait_warp(full0 + 8 * stage, phase, p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
      if (!ok) break;
      const TileRec rec = tile_rec[stage];
      if (rec.flags & (kRecFirst | kRecEnd)) {
        // Wait until the epilogue has drained this accumulator.
        buf = tcount % NBUF;
        const bool r = mbar_wait_warp(acce0 + 8 * buf, ((tcount / NBUF) & 1u) ^ 1u, p.wait_limit_ns);
        ok = __shfl_sync(0xffffffffu, r && !*abort_flag, 0);
        if (!ok) break;
        tc_fence_after_sync();
        seg_flags = rec.flags & (kRecTileFirst | kRecAtF0);
      }
      if (rec.flags & kRecEnd) {
        if (leader) {
          acc_rec[buf].flags = kRecEnd;
          mbar_arrive(accf0 + 8 * buf);
          mbar_arrive(accf0 + 8 * buf);
        }
        break;
      }
      {  // converged: one elected lane issues each MMA and commit
        if (!(rec.flags & kRecEmpty)) {
          tc_fence_after_sync();
          const int nmma = min(C_::kMmas, (p.N - rec.nt * BN + C_::kNmma - 1) / C_::kNmma);
          const uint32_t acc = tmem + buf * C_::kAccCols;
          const bool first = (rec.flags & kRecFirst) != 0;
          // Descriptors of the stage's first block; every other operand is a
          // fixed byte offset from them (smem_desc_add).
          const uint32_t st0 = smem_addr(smem + stage * C_::kStageBytes);
          const uint64_t adesc0 = smem_desc_sw128(st0, 16, 1024);                    // block: A, K-major
          const uint64_t bdesc0 = smem_desc_sw128(st0 + kBlkBytes, kChunkBytes, 1024);  // B tile: MN-major
#pragma unroll
          for (int b = 0; b < KB; ++b) {
            if (b < rec.nblk) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t adesc = smem_desc_add(adesc0, b * C_::kSubBytes + kk * 32);
                const uint32_t acc_in = (first && b == 0 && kk == 0) ? 0u : 1u;  // the tile's first step overwrites
#pragma unroll
                for (int m = 0; m < C_::kMmas; ++m) {
                  if (m < nmma) {
                    const uint64_t bdesc = smem_desc_add(
                        bdesc0, b * C_::kSubBytes + m * (C_::kNmma / 64) * kChunkBytes + kk * 2048);
                    if constexpr (C_::kWS)
                      umma_ws_f16_elect(acc, adesc, bdesc, idesc, acc_in);
                    else
                      umma_f16_elect(acc + m * C_::kNmma, adesc, bdesc, idesc, acc_in);
                  }
                }
              }
            }
          }
        }
        umma_commit_elect(empty0 + 8 * stage);  // frees the stage once these MMAs have read it
        if (rec.flags & kRecLast) {
          if (leader) {
            acc_rec[buf].br = rec.br;
            acc_rec[buf].nt = rec.nt;
            acc_rec[buf].flags = (rec.flags & (kRecEmpty | kRecTileLast)) | seg_flags;
            mbar_arrive(accf0 + 8 * buf);  // releases the record
          }
          umma_commit_elect(accf0 + 8 * buf);  // arrives when the tile's MMAs are done
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
        for (int b = 0; b < NBUF; ++b) {
          mbar_arrive(accf0 + 8 * b);
          mbar_arrive(accf0 + 8 * b);
        }
      }
    }
    grid_launch_dependents();  // every MMA is issued: the next kernel may be scheduled
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM sub-partition s = w % 4; lane t holds one row of C
    // (see Cfg for which rows and columns).  Its 16-column pieces go to the
    // warp's staging area as store boxes in the swizzled layout the TMA store
    // reads.  Each batch of TMEM loads is issued before the previous batch is
    // written to shared memory, so the load latency overlaps that work.
    const int sp = warp & 3;
    uint8_t *stg = staging + (warp - kEpiWarp0) * C_::kWarpStaging;
    const uint32_t stg_addr = smem_addr(stg);
    // 16-byte unit u of box row t is stored at unit u ^ row_sw
    const uint32_t row_sw = static_cast<uint32_t>(C_::kWS ? (lane >> 1) & 3 : lane & 7);
    const bool row_lane = lane < C_::kWarpRows;
    uint32_t tcount = 0;
    while (true) {
      const uint32_t buf = tcount % NBUF;
      const bool r = mbar_wait_warp(accf0 + 8 * buf, (tcount / NBUF) & 1u, p.wait_limit_ns);
      if (!__shfl_sync(0xffffffffu, r && !*abort_flag, 0)) {
        if (lane == 0 && !r) {
          atomicOr(p.status, kDevTimeout);
          *abort_flag = 1;
        }
        break;
      }
      const int32_t flags = acc_rec[buf].flags;
      if (flags & kRecEnd) break;
      if ((flags & kRecWhole) != kRecWhole) {
        // A segment of a tile cut between CTAs (split schedule): its fp32
        // partial sums go to this CTA's workspace slot (64 rows x BN columns,
        // row-major) for split_reduce_kernel, with a record naming the tile.
        const int slot = 2 * static_cast<int>(blockIdx.x) + ((flags & kRecAtF0) ? 0 : 1);
        float *ws = p.workspace + static_cast<int64_t>(slot) * kBcsrSlotFloats;
        const int br_s = acc_rec[buf].br;
        const int nt_s = acc_rec[buf].nt;
        const int row = (C_::kWS ? (sp & 1) * 32 : sp * 16) + lane;
        const int col0 = C_::kWS ? (sp >> 1) * C_::kWarpCols : 0;
        tc_fence_after_sync();
        const uint32_t tbase = tmem + (static_cast<uint32_t>(sp * 32) << 16) + buf * C_::kAccCols;
#pragma unroll 1
        for (int g = 0; g < C_::kWarpCols / 16; ++g) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tbase + g * 16, v);
          tmem_ld_wait();
          if (row_lane && nt_s * BN + col0 + g * 16 < p.N) {
            float4 *dst = reinterpret_cast<float4 *>(ws + row * BN + col0 + g * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if (warp == kEpiWarp0)
            p.partials[slot] = PartialRec{br_s, nt_s,
                                          ((flags & kRecTileFirst) ? kStageFirst : 0) |
                                              ((flags & kRecTileLast) ? kStageLast : 0),
                                          0};
          mbar_arrive(acce0 + 8 * buf);
        }
        ++tcount;
        continue;
      }
      const bool zero = (flags & kRecEmpty) != 0;
      const int row0 = acc_rec[buf].br * kBlk + (C_::kWS ? (sp & 1) * 32 : sp * 16);
      const int n0 = acc_rec[buf].nt * BN + (C_::kWS ? (sp >> 1) * C_::kWarpCols : 0);  // this warp's first column
      const int ncg = max(0, min(C_::kWarpCols / 16, (p.N - n0 + 15) / 16));  // 16-column groups holding C
      tc_fence_after_sync();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(sp * 32) << 16) + buf * C_::kAccCols;
      // kBatch 16-column groups starting at group g0 -> registers
      auto load_batch = [&](int g0, uint32_t (&v)[C_::kBatch][16]) {
#pragma unroll
        for (int g = 0; g < C_::kBatch; ++g) {
          if (g0 + g < ncg && !zero) {
            tmem_ld_32x32b_x16(tbase + (g0 + g) * 16, v[g]);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[g][i] = 0u;
          }
        }
      };
      // registers -> staging part `pst` (gl0: first group of the part)
      auto store_batch = [&](uint8_t *pst, int g0, int gl0, const uint32_t (&v)[C_::kBatch][16]) {
        if (row_lane) {
#pragma unroll
          for (int g = 0; g < C_::kBatch; ++g) {
            const int col = (g0 + g - gl0) * 16;  // column within the part
            uint8_t *row_base = pst + (col / C_::kBoxCols) * kBoxBytes + lane * C_::kRowBytes;
            const uint32_t u0 = static_cast<uint32_t>((col % C_::kBoxCols) * C_::kOutBytes / 16);
            if constexpr (OUT_BF16) {
              uint32_t w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const __nv_bfloat162 h =
                    __floats2bfloat162_rn(__uint_as_float(v[g][2 * i]), __uint_as_float(v[g][2 * i + 1]));
                w[i] = *reinterpret_cast<const uint32_t *>(&h);
              }
              *reinterpret_cast<uint4 *>(row_base + (((u0 + 0) ^ row_sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4 *>(row_base + (((u0 + 1) ^ row_sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4 *>(row_base + (((u0 + q) ^ row_sw) << 4)) =
                    make_uint4(v[g][4 * q], v[g][4 * q + 1], v[g][4 * q + 2], v[g][4 * q + 3]);
            }
          }
        }
      };
#pragma unroll
      for (int part = 0; part < PARTS; ++part) {
        const int gl0 = part * C_::kPartGroups;
        uint8_t *pst = stg + (part & 1) * C_::kPartBytes;
        // this part's staging buffer is free once at most one store group
        // (the other part's) is still reading shared memory
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint32_t va[C_::kBatch][16], vb[C_::kBatch][16];
        constexpr int kB = C_::kBatch;
        load_batch(gl0, va);
#pragma unroll
        for (int b = 0; b < C_::kBatches; b += 2) {
          tmem_ld_wait();
          if (b + 1 < C_::kBatches) load_batch(gl0 + (b + 1) * kB, vb);
          store_batch(pst, gl0 + b * kB, gl0, va);
          if (b + 1 < C_::kBatches) {
            tmem_ld_wait();
            if (b + 2 < C_::kBatches) load_batch(gl0 + (b + 2) * kB, va);
            store_batch(pst, gl0 + (b + 1) * kB, gl0, vb);
          }
        }
        if (part == PARTS - 1) tc_fence_before_sync();  // this warp's reads of the accumulator are complete
        fence_proxy_async_smem();               // the staging writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0) {
          if (part == PARTS - 1) mbar_arrive(acce0 + 8 * buf);
          if (row0 < p.M) {
            for (int b = 0; b < C_::kPartBoxes; ++b) {
              const int x = n0 + part * C_::kPartCols + b * C_::kBoxCols;
              if (x < p.N) tma_store_2d(&tmC, smem_addr(pst) + b * kBoxBytes, x, row0);
            }
          }
          bulk_commit_group();
        }
      }
      ++tcount;
    }
    (void)stg_addr;
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C_::kTmemCols);
  }
}

template <int BN, int Q, int NBUF, int PARTS, int MINB, int PW, int KB, bool IN_BF16, bool OUT_BF16>
cudaError_t launch_variant(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                           const BcsrParams &p, cudaStream_t stream) {
  using C_ = Cfg<BN, Q, NBUF, PARTS, MINB, PW, KB, OUT_BF16>;
  auto kern = bcsr_spmm_kernel<BN, Q, NBUF, PARTS, MINB, PW, KB, IN_BF16, OUT_BF16>;
  static std::atomic<uint64_t> smem_set{0};  // per instantiation, one bit per device
  cudaError_t e = set_smem_limit_once(kern, C_::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  int64_t grid;
  if (p.split_grid > 0) {
    grid = p.split_grid;
  } else {
    const int64_t tiles = static_cast<int64_t>(p.n_block_rows) * ((p.N + BN - 1) / BN);
    const int64_t cap = p.max_ctas > 0 ? p.max_ctas : static_cast<int64_t>(MINB) * p.num_sms;
    grid = tiles < cap ? tiles : cap;
  }
  kern<<<static_cast<unsigned>(grid), C_::kThreads, C_::kSmemBytes, stream>>>(tmA, tmB, tmC, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.split_grid == 0) return e;
  return launch_split_reduce<kBlk, OUT_BF16>(p.partials, p.workspace, kBcsrSlotFloats, BN, p.C, p.M, p.N,
                                             static_cast<int32_t>(grid), BN, stream);
}

template <int BN, int Q, int NBUF, int PARTS, int MINB, int PW, int KB, bool OUT_BF16>
cudaError_t launch_in(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const BcsrParams &p,
                      bool in_bf16, cudaStream_t s) {
  return in_bf16 ? launch_variant<BN, Q, NBUF, PARTS, MINB, PW, KB, true, OUT_BF16>(tmA, tmB, tmC, p, s)
                 : launch_variant<BN, Q, NBUF, PARTS, MINB, PW, KB, false, OUT_BF16>(tmA, tmB, tmC, p, s);
}

}  // namespace

int bcsr_tile_cols(int64_t N) { return bcsr_wide_tiles(N) ? 256 : 128; }

cudaError_t launch_bcsr(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const BcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t stream) {
  if (p.n_block_rows == 0 || p.N == 0) return cudaSuccess;
  // N <= 128: 128-column tiles (one plain MMA of N = 128 per k step), two
  // accumulators; one CTA per SM with four stages of two blocks each (the
  // MMA thread's fixed cost per stage, ~600 cycles besides the MMAs, bounds
  // these shapes; two blocks per stage cut the 8192^2 sweeps by 20-24 %), or,
  // on the split schedule, two CTAs per SM with three one-block stages.
  // Wider (bcsr_wide_tiles): 256-column tiles, one weight-stationary MMA of
  // N = 256 per k step, two accumulators of 128 TMEM columns; with at least
  // two tiles per SM (or on the split schedule) two CTAs share each SM (two
  // stages each), so one CTA's barrier handshakes overlap the other's MMAs
  // and loads; with fewer tiles one CTA per SM runs four stages (two blocks
  // per stage measured no faster there).  Epilogue parts are one 32-row x
  // 64-byte store box (32 bf16 or 16 fp32 columns).
  if (!bcsr_wide_tiles(p.N)) {
    if (p.split_grid > 0)
      return out_bf16 ? launch_in<128, 3, 2, 2, 2, 1, 1, true>(tmA, tmB, tmC, p, in_bf16, stream)
                      : launch_in<128, 3, 2, 2, 2, 1, 1, false>(tmA, tmB, tmC, p, in_bf16, stream);
    return out_bf16 ? launch_in<128, 4, 2, 2, 1, 1, 2, true>(tmA, tmB, tmC, p, in_bf16, stream)
                    : launch_in<128, 4, 2, 2, 1, 1, 2, false>(tmA, tmB, tmC, p, in_bf16, stream);
  }
  const int64_t tiles = static_cast<int64_t>(p.n_block_rows) * ((p.N + 255) / 256);
  if (tiles < 2ll * p.num_sms && p.split_grid == 0)
    return out_bf16 ? launch_in<256, 4, 2, 4, 1, 1, 1, true>(tmA, tmB, tmC, p, in_bf16, stream)
                    : launch_in<256, 4, 2, 8, 1, 1, 1, false>(tmA, tmB, tmC, p, in_bf16, stream);
  return out_bf16 ? launch_in<256, 2, 2, 4, 2, 1, 1, true>(tmA, tmB, tmC, p, in_bf16, stream)
                  : launch_in<256, 2, 2, 8, 2, 1, 1, false>(tmA, tmB, tmC, p, in_bf16, stream);
}

}  // namespace spmm
