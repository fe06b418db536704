// wcsr_kernel.cu -- WCSR SpMM for sm_103a.
//
// Method: "AsyncSparse", Section III-B (a window's packed value tile is
// contiguous; the rows of B it multiplies are fetched
// through window_col_idx by all threads, written to shared memory with the
// 128-byte swizzle applied by hand) and Section III-C (task decomposition so
// that long windows do not serialise on one CTA).
//
// Work list: every window is cut into stages of at most 64 packed columns,
// listed in window order (a window without columns has one empty stage).  The
// T = stages x column-tiles work items are cut into G equal contiguous chunks,
// chunk c = [T*c/G, T*(c+1)/G), and the grid has one CTA per chunk.  By
// default G is the number of CTAs that fit (two per SM) and each CTA runs its
// own chunk: every CTA gets the same number of stages whatever the window
// lengths, and the column indices it reads are contiguous.  With p.dynamic
// (Section V's future work on Blackwell) G is about four times that, and a
// CTA that finishes a chunk cancels the launch of a CTA that has not started
// and takes over its chunk (cluster launch control).  A window whose stages
// are cut by a chunk boundary is finished by a second kernel: each chunk's
// fp32 partial sums of its first and last window go to two workspace slots,
// and the slot holding the window's first stage adds the slots of the
// following chunks in chunk order (the paper adds split partials with
// atomicAdd; the fixed order here makes results bitwise reproducible).
//
// The product is computed transposed: the 128 columns of an accumulator are
// the MMA's M (TMEM lanes) and the 16 rows of a window are the MMA's N.
//
// Only the producer warps read global memory.  Each stage is one record in
// global memory: its 2 KB value tile, 64 column indices and a descriptor.  A
// producer warp fetches the index part of its items' records (272 bytes) by
// TMA bulk copies into a per-warp ring kIdxLead of its items ahead, so it
// reads an item's indices from shared memory without waiting; when it starts
// the item it has the value tile copied into the item's stage by TMA and
// copies the item's rows of B with cp.async, all completing on the stage's
// barrier.  The MMA thread learns a stage's shape from a record the producer
// writes to shared memory, and the epilogue learns a window's identity from a
// record the MMA thread writes, so neither waits on a global load.
//
// PW + 5 warps (two CTAs per SM, so one CTA's barrier handshakes and MMA
// issue stalls overlap the other's work):
//   warps 0..PW-1  producers, in groups of WPG warps; group g owns the work
//                  items g, g + PW/WPG, ... of the CTA's sequence, and each
//                  warp of a group copies its share of an item's 64 B rows
//                  with 16-byte cp.async (one B row, 512 B, per warp
//                  instruction at BN = 256); every lane ends the item with
//                  cp.async.mbarrier.arrive.noinc, so producers never block
//                  on their own copies and one warp's barrier handling
//                  overlaps another's copies
//   warp PW        TMEM allocator and MMA issuer; fences the generic proxy
//                  against the async proxy before reading a stage
//   warps PW+1..   epilogue (warp w reads TMEM sub-partition w % 4), four
//                  accumulator buffers in TMEM rotate between windows
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "split_reduce.cuh"

namespace spmm {
namespace {

constexpr int kH = 16;                       // window height
constexpr int kKC = 64;                      // packed columns per stage
constexpr int kValBytes = kH * kKC * 2;      // 2 KB value tile per stage
constexpr int kMetaBytes = kWcsrPackBytes - kWcsrPackIdxOff;  // a stage record's indices + descriptor
constexpr int kChunkBytes = kKC * 64 * 2;    // 64 gathered rows x 64 columns
constexpr int kEpiWarps = 4;
constexpr int kAccBufs = 4;
constexpr int kRespSlots = 4;  // cluster-launch-control answers in flight (dynamic schedule)

// Stage record flags besides kStageFirst / kStageLast (the window's first and
// last stage): the first and last work item of a chunk, and the end of the
// CTA's work.
constexpr int32_t kRecChunkFirst = 4;
constexpr int32_t kRecChunkLast = 8;
constexpr int32_t kRecEnd = 16;

// A producer fetches the column-index record of its items this many of its
// own items ahead (a small TMA bulk copy into a per-warp ring), so reading an
// item's indices never waits on memory; the item's 2 KB value tile is fetched
// into the item's stage together with the gather (and brought into L2 when
// its index record is fetched).
constexpr int kIdxLead = 4;

// NACC accumulators of 128 columns, Q stages, PW producer warps in groups of
// WPG (the WPG warps of a group copy disjoint row ranges of the same work
// items: a warp's cp.async issue rate is limited, about 13 bytes per clock on
// GB300, so the gather rate of an SM grows with its copying warps up to about
// 12), MINB CTAs per
// SM, ILEAD index-record slots per producer warp (0: indices are read from
// global memory, the no-allocation variant).  A stage holds an item's gathered
// B rows and its value tile.
template <int NACC, int Q, int PW, int WPG, int MINB, int ILEAD>
struct Cfg {
  static constexpr int kGroups = PW / WPG;                  // producer groups: group g owns items g, g + kGroups, ...
  static constexpr int kMmaWarp = PW;                        // warps 0..PW-1 produce, PW issues MMAs
  static constexpr int kThreads = 32 * (PW + 1 + kEpiWarps);
  static constexpr int kBN = 128 * NACC;
  static constexpr int kChunks = 2 * NACC;
  static constexpr int kGatherBytes = kChunks * kChunkBytes;  // gathered B rows
  static constexpr int kStageBytes = kGatherBytes + kValBytes;
  static constexpr int kAccCols = kH * NACC;                     // TMEM columns per accumulator buffer
  static constexpr int kTmemCols = kAccBufs * kAccCols <= 32 ? 32 : (kAccBufs * kAccCols <= 64 ? 64 : 128);
  static constexpr int kIdxRing = (PW * ILEAD * kMetaBytes + 1023) / 1024 * 1024;
  static constexpr int kBars = 2 * Q + 2 * kAccBufs + 1 + PW * ILEAD + kRespSlots;
  static constexpr int kMiscBytes = 2048;  // launch-control answers, barriers, TMEM address, records between roles
  static constexpr int kSmemBytes = Q * kStageBytes + kIdxRing + kMiscBytes + 1024;
  static_assert(kStageBytes % 1024 == 0 && kGatherBytes % 1024 == 0, "MMA operands need 1024-byte alignment");
  // A producer's wait for stage (it % Q) to be free is a parity wait on the
  // MMA commit of item it - Q; it is only unambiguous if the commit of item
  // it - 2Q has already been seen, which the warp's wait for its previous item
  // (it - kGroups) guarantees when kGroups <= Q.  With more producer groups
  // than stages a warp could run two phases ahead, pass the wait early and
  // overwrite a stage still in use.
  static_assert(PW % WPG == 0 && 64 % WPG == 0 && WPG <= 4, "producer groups");
  static_assert(kGroups <= Q, "more producer groups than stages");
  static_assert(kRespSlots * 16 + kBars * 8 + 16 + Q * 32 + kAccBufs * 32 <= kMiscBytes, "barrier area");
  static_assert(kSmemBytes <= 227 * 1024 && MINB * (kSmemBytes + 1024) <= 228 * 1024, "shared memory");
  static_assert(MINB * kTmemCols <= 512, "TMEM");
  static_assert(kAccBufs * kAccCols <= kTmemCols, "accumulator buffers exceed the TMEM allocation");
};

// Shared-memory records passed between roles.
struct StageRec {   // producer -> MMA, one per ring stage
  int32_t ncols;
  int32_t flags;    // kStageFirst | kStageLast | kRecChunkFirst | kRecChunkLast | kRecEnd
  int32_t window;
  int32_t tile;
  int32_t chunk;    // the chunk the item belongs to (its partial-sum slots are 2 chunk, 2 chunk + 1)
  int32_t pad_[3];
};
struct SegRec {     // MMA -> epilogue, one per accumulator buffer
  int32_t window;   // -1: no more segments
  int32_t tile;
  int32_t flags;    // kStageFirst | kStageLast of the window, as covered by this CTA
  int32_t zero;     // no MMA was issued (a window without columns)
  int32_t slot;     // workspace slot for a partial segment
  int32_t pad_[3];
};

// NOALLOC: the variant behind spmm_wcsr_run_noalloc -- the stage count is
// read from device memory (the stage list is built on the device), CTAs
// beyond the number of work items leave at once, and column indices are read
// from window_col_idx at each stage's first packed column.
template <int NACC, int Q, int PW, int WPG, int MINB, bool IN_BF16, bool OUT_BF16, bool NOALLOC = false,
          bool DYN = false>
__global__ void __launch_bounds__(32 * (PW + 1 + kEpiWarps), MINB)
    wcsr_spmm_kernel(const WcsrParams p) {
  constexpr int kILead = NOALLOC ? 0 : kIdxLead;
  using C_ = Cfg<NACC, Q, PW, WPG, MINB, kILead>;
  static_assert(!NOALLOC || WPG == 1, "the no-allocation variant copies each item with one warp");
  constexpr int kMmaWarp = C_::kMmaWarp;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *iring = smem + Q * C_::kStageBytes;  // per producer warp: kILead index records of kMetaBytes
  uint8_t *resp = iring + C_::kIdxRing;         // kRespSlots x 16-byte launch-control answers
  uint64_t *bars = reinterpret_cast<uint64_t *>(resp + 16 * kRespSlots);
  // bars: full[Q], empty[Q], acc_full[kAccBufs], acc_empty[kAccBufs], drain, ifull[PW][kILead],
  // resp[kRespSlots]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C_::kBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  StageRec *stage_rec = reinterpret_cast<StageRec *>(tmem_slot + 4);        // [Q]
  volatile SegRec *seg_rec = reinterpret_cast<volatile SegRec *>(stage_rec + Q);  // [kAccBufs]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_col_tiles = (p.N + C_::kBN - 1) / C_::kBN;
  const int64_t n_stages = NOALLOC ? *p.n_stages_dev : p.n_stages;
  const int64_t total = n_stages * n_col_tiles;
  const int64_t grid = NOALLOC ? (total < gridDim.x ? total : gridDim.x) : gridDim.x;
  if (NOALLOC && blockIdx.x >= grid) {
    if (threadIdx.x == 0) {
      p.partials[2 * blockIdx.x] = PartialRec{-1, 0, 0, 0};
      p.partials[2 * blockIdx.x + 1] = PartialRec{-1, 0, 0, 0};
    }
    return;
  }
  const int64_t f0 = total * blockIdx.x / grid;
  const int64_t f1 = total * (blockIdx.x + 1) / grid;

  const uint32_t full0 = smem_addr(&bars[0]);
  const uint32_t empty0 = smem_addr(&bars[Q]);
  const uint32_t accf0 = smem_addr(&bars[2 * Q]);
  const uint32_t acce0 = smem_addr(&bars[2 * Q + kAccBufs]);
  const uint32_t drain_bar = smem_addr(&bars[2 * Q + 2 * kAccBufs]);
  const uint32_t ifull0 = smem_addr(&bars[2 * Q + 2 * kAccBufs + 1]);
  const uint32_t respb0 = smem_addr(&bars[2 * Q + 2 * kAccBufs + 1 + PW * kILead]);
  const uint32_t resp0 = smem_addr(resp);

  if (threadIdx.x == 0) {
    for (int q = 0; q < Q; ++q) {
      // 32 cp.async lane arrivals per warp of the item's group (gathered rows;
      // the value tile too in the no-allocation variant) + one arrive of the
      // group's first warp, which releases the stage record and expects the
      // value tile's TMA bytes
      mbar_init(full0 + 8 * q, 1 + 32 * WPG);
      mbar_init(empty0 + 8 * q, 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(accf0 + 8 * b, 2);  // the MMA commit + the MMA thread's arrive (segment record)
      mbar_init(acce0 + 8 * b, kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int v = 0; v < PW * kILead; ++v) mbar_init(ifull0 + 8 * v, 1);  // lane 0's expect_tx arrive
    for (int v = 0; v < kRespSlots; ++v) mbar_init(respb0 + 8 * v, 1);   // expect_tx arrive + 16-byte answer
    *abort_flag = 0;
    fence_barrier_init();
    if (NOALLOC) {  // partial-sum records of this CTA (overwritten below when used)
      p.partials[2 * blockIdx.x] = PartialRec{-1, 0, 0, 0};
      p.partials[2 * blockIdx.x + 1] = PartialRec{-1, 0, 0, 0};
    }
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
    // ------------------------------------------------------------ producers
    const uint16_t *Bp = reinterpret_cast<const uint16_t *>(p.B);
    constexpr int kStep = PW;                 // (no-allocation variant: one warp per group)
    constexpr int G = C_::kGroups;
    const int grp = warp / WPG, sub = warp % WPG;
    const int rbeg = sub * (64 / WPG), rend = rbeg + 64 / WPG;  // this warp's rows of every item
    // The B rows of one work item -> stage `st` with 16-byte cp.async; lo /
    // hi hold the item's column indices for positions lane and 32 + lane.
    // Only the 16-byte units of the tile's live columns (below N) are copied:
    // output column m of the transposed product depends on gathered column m
    // alone, and columns at or past N are never stored, so whatever the stage
    // holds there does not matter.  A padding position (index -1) is
    // zero-filled, since its zero values multiply it.  Each warp instruction
    // copies 32 (row, unit) pairs, U units per row (U = live units rounded up
    // to a power of two), so at small N a stage costs a few instructions.
    // Only rows [rbeg, rend) are copied by this warp.
    auto gather = [&](uint32_t st, int n0, int ncols, int32_t lo, int32_t hi) {
      const int rlim = min(ncols, rend);
      const int live_units = (min(C_::kBN, p.N - n0) + 7) >> 3;  // 1 .. 16 * NACC
      if (live_units == 16 * NACC) {
        // every unit live: the row layout is fixed at compile time (one B row
        // per instruction at BN = 256, two at BN = 128)
        constexpr int kRowsPerInst = 2 / NACC;
        const int v = lane & (16 * NACC - 1);
        const int rl = lane / (16 * NACC);
        const int n = n0 + v * 8;
        const uint32_t dst_col = (v >> 3) * kChunkBytes;
        const uint32_t uu = static_cast<uint32_t>(v & 7);
        for (int r0 = rbeg; r0 < rlim; r0 += 16) {
          const int32_t src = r0 < 32 ? lo : hi;
          constexpr int kInst = 16 / kRowsPerInst;
          int32_t col[kInst];
#pragma unroll
          for (int j = 0; j < kInst; ++j) col[j] = __shfl_sync(0xffffffffu, src, (r0 + kRowsPerInst * j + rl) & 31);
#pragma unroll
          for (int j = 0; j < kInst; ++j) {
            const int r = r0 + kRowsPerInst * j + rl;
            // caller-supplied indices (no-allocation variant) are clamped to B's rows
            const bool live = col[j] >= 0 && (!NOALLOC || col[j] < p.K);
            cp_async_16(st + dst_col + r * 128 + ((uu ^ static_cast<uint32_t>(r & 7)) << 4),
                        live ? static_cast<const void *>(Bp + static_cast<int64_t>(col[j]) * p.N + n)
                             : static_cast<const void *>(Bp),
                        live ? 16u : 0u);
          }
        }
        return;
      }
      const int sh = 32 - __clz(live_units - 1);                 // log2 of U (0 for one unit)
      const int rsh = 5 - sh;                                    // log2 of rows per instruction
      const int i_beg = rbeg >> rsh;                             // instructions holding rows [rbeg, rlim)
      const int i_end = (rlim + (1 << rsh) - 1) >> rsh;
      const int r_lane = lane >> sh;                             // this lane's row within an instruction
      const int u = lane & ((1 << sh) - 1);                      // this lane's unit within its row
      const int n = n0 + u * 8;
      const bool u_live = n < p.N;
      const uint32_t dst_u = (u >> 3) * kChunkBytes;
      const uint32_t uu = static_cast<uint32_t>(u & 7);
      // 16 instructions at a time: their shuffles issue back to back instead
      // of each copy waiting for the last
      for (int i0 = i_beg; i0 < i_end; i0 += 16) {
        int32_t col[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int rb = (i0 + j) << rsh;  // first row of instruction i0 + j
          col[j] = __shfl_sync(0xffffffffu, rb < 32 ? lo : hi, (rb + r_lane) & 31);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = ((i0 + j) << rsh) + r_lane;
          if (i0 + j < i_end && u_live && r >= rbeg && r < rlim) {
            // caller-supplied indices (no-allocation variant) are clamped to B's rows
            const bool live = col[j] >= 0 && (!NOALLOC || col[j] < p.K);
            cp_async_16(st + dst_u + r * 128 + ((uu ^ static_cast<uint32_t>(r & 7)) << 4),
                        live ? static_cast<const void *>(Bp + static_cast<int64_t>(col[j]) * p.N + n)
                             : static_cast<const void *>(Bp),
                        live ? 16u : 0u);
          }
        }
      }
    };
    // The end of the CTA's work: the group owning CTA-local item it_end (the
    // one after the last, group it_end % G) passes an end record to the MMA
    // warp through stage it_end % Q.
    auto send_end = [&](int64_t it_end) -> bool {
      const uint32_t stage = static_cast<uint32_t>(it_end % Q);
      const uint32_t phase = static_cast<uint32_t>((it_end / Q) & 1);
      bool r = mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns);
      r = __shfl_sync(0xffffffffu, r && !*abort_flag, 0);
      if (!r) return false;
      if (lane == 0 && sub == 0) {
        stage_rec[stage] = StageRec{0, kRecEnd, -1, 0, 0, {0, 0, 0}};
        mbar_arrive(full0 + 8 * stage);
      }
      cp_async_arrive_noinc(full0 + 8 * stage);
      return true;
    };
    if constexpr (NOALLOC) {
      // Caller-owned arrays: the stage list built on the device, the column
      // indices read at each stage's first packed column, and the values
      // copied from the row-major [16][P_total] array (swizzled here) into the
      // item's stage with the gather.  Work items of this warp: f = f0 + warp
      // + PW*i.  Descriptors are loaded four of the warp's items ahead and
      // column indices two items ahead, into ring slots chosen by the
      // (unrolled) item position, so a register is only read long after its
      // load was issued.
      const int4 *stg = reinterpret_cast<const int4 *>(p.stages);
      int4 ring_d[4];
      int32_t ring_lo[2], ring_hi[2];
      auto load_d = [&](int64_t fi) -> int4 { return fi < f1 ? stg[fi % n_stages] : make_int4(0, -1, 0, 0); };
      auto load_idx = [&](int k, const int4 &dd) {
        ring_lo[k] = lane < dd.z ? p.window_col_idx[static_cast<int64_t>(dd.x) + lane] : -2;
        ring_hi[k] = lane + 32 < dd.z ? p.window_col_idx[static_cast<int64_t>(dd.x) + 32 + lane] : -2;
      };
      // value tile of descriptor dd -> the stage's value area (zeros past
      // ncols: the MMA reads whole 16-column k-steps only up to ncols)
      auto copy_vals = [&](uint32_t vdst, const int4 &dd) {
        if (dd.z > 0) {
          const uint16_t *Vp = reinterpret_cast<const uint16_t *>(p.values);
          const uint32_t u = static_cast<uint32_t>(lane & 7);
          const int64_t pcol = static_cast<int64_t>(dd.x) + u * 8;
          const bool in = pcol < p.P_total;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = (lane >> 3) + 4 * q;
            cp_async_16(vdst + r * 128 + ((u ^ static_cast<uint32_t>(r & 7)) << 4),
                        in ? static_cast<const void *>(Vp + r * p.P_total + pcol) : static_cast<const void *>(Vp),
                        in ? 16u : 0u);
          }
        }
      };
      int64_t f = f0 + warp;
#pragma unroll
      for (int u = 0; u < 4; ++u) ring_d[u] = load_d(f + u * kStep);
      load_idx(0, ring_d[0]);
      load_idx(1, ring_d[1]);
      bool ok = true;
      for (; f < f1 && ok; f += 4 * kStep) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t fi = f + u * kStep;
          if (fi >= f1 || !ok) break;
          const int4 d = ring_d[u];
          const int32_t lo = ring_lo[u & 1], hi = ring_hi[u & 1];
          load_idx(u & 1, ring_d[(u + 2) & 3]);
          ring_d[u] = load_d(fi + 4 * kStep);
          const int64_t it = fi - f0;
          const uint32_t stage = static_cast<uint32_t>(it % Q);
          const uint32_t phase = static_cast<uint32_t>((it / Q) & 1);
          ok = mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns);
          ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
          if (!ok) break;
          const uint32_t st = smem_addr(smem + stage * C_::kStageBytes);
          const uint32_t fb = full0 + 8 * stage;
          const int tile = static_cast<int>(fi / n_stages);
          if (lane == 0) {  // released by this arrive
            const int32_t fl = d.w | (fi == f0 ? kRecChunkFirst : 0) | (fi == f1 - 1 ? kRecChunkLast : 0);
            stage_rec[stage] = StageRec{d.z, fl, d.y, tile, static_cast<int32_t>(blockIdx.x), {0, 0, 0}};
            mbar_arrive(fb);
          }
          copy_vals(st + C_::kGatherBytes, d);
          gather(st, tile * C_::kBN, d.z, lo, hi);
          cp_async_arrive_noinc(fb);
        }
      }
      if (ok && (f1 - f0) % PW == warp) ok = send_end(f1 - f0);
      cp_async_wait_all();
      if (!ok && lane == 0) {
        atomicOr(p.status, kDevTimeout);
        *abort_flag = 1;
      }
    } else {
      // Every stage is one record in global memory (its value tile, its 64
      // column indices and its descriptor).
      //
      // Chunks: the CTA's work is a sequence of chunks, chunk id being the
      // work items [T*id/G, T*(id+1)/G) (G = gridDim.x).  The first is chunk
      // blockIdx.x; with p.dynamic every further one is a CTA of this grid
      // that had not started yet, cancelled through cluster launch control
      // and taken over here (the paper's future-work dynamic scheduling,
      // Section V); without it the CTA has just its own chunk.  Warp 0
      // requests the next chunk when it learns of one, into answer slot
      // (ordinal % kRespSlots); every producer warp reads the same answers,
      // so all of them see the same sequence.  CTA-local item it (0, 1, ...
      // across the chunks) belongs to producer group it % G and stage it % Q.
      //
      // Each warp fetches the index part of its group's item j's record (272 bytes)
      // kILead of its items ahead into slot j % kILead of its ring, and when
      // it starts item j it reads the indices from there (the slot is then
      // refilled), waits for the item's stage to be free, has the value tile
      // copied into the stage by TMA and copies the item's rows of B with
      // cp.async.  Chunks hold at least 32 items (at most 16 of a warp's items
      // apart are live at once), so the answer slots and the four remembered
      // chunks are never overwritten while a warp still needs them.
      const uint8_t *pack = reinterpret_cast<const uint8_t *>(p.stage_pack);
      uint8_t *ring = iring + warp * kILead * kMetaBytes;
      const uint32_t ifull_w = ifull0 + 8 * (warp * kILead);
      const int64_t n_chunks = gridDim.x;
      struct Chunk {
        int64_t lbase, len, g0;  // first CTA-local item, items, first work item
        int32_t id;
      };
      // the last four chunks learned (the static schedule has one)
      constexpr int kKn = DYN ? 4 : 1;
      Chunk kn[kKn] = {};
      int nk = 0;               // chunks learned
      bool no_more = false;     // the chunk after the last learned one does not exist
      int64_t l_end = 0;        // CTA-local items in all (once no_more)
      int64_t n_req = 0, n_read = 0;  // warp 0: answers requested / read
      bool ok = true;
      // Learns chunk nk (false: a wait ran out).
      auto learn_next = [&]() -> bool {
        int32_t id = -1;
        if (nk == 0) {
          id = static_cast<int32_t>(blockIdx.x);
        } else if (DYN) {
          const uint32_t sl = static_cast<uint32_t>((nk - 1) % kRespSlots);
          bool r = mbar_wait_warp(respb0 + 8 * sl, static_cast<uint32_t>(((nk - 1) / kRespSlots) & 1),
                                  p.wait_limit_ns);
          r = __shfl_sync(0xffffffffu, r && !*abort_flag, 0);
          if (!r) return false;
          uint32_t x = 0;
          const bool got = clc_query(resp0 + 16 * sl, x);
          ++n_read;
          id = got ? static_cast<int32_t>(x) : -1;
        }
        const int64_t lb = nk ? kn[(nk - 1) & (kKn - 1)].lbase + kn[(nk - 1) & (kKn - 1)].len : 0;
        if (id < 0) {
          no_more = true;
          l_end = lb;
          return true;
        }
        Chunk c;
        c.id = id;
        c.g0 = total * id / n_chunks;
        c.len = total * (id + 1) / n_chunks - c.g0;
        c.lbase = lb;
        kn[nk & (kKn - 1)] = c;
        if (DYN && warp == 0) {
          if (lane == 0) {
            const uint32_t sl = static_cast<uint32_t>(nk % kRespSlots);
            mbar_arrive_expect_tx(respb0 + 8 * sl, 16);
            clc_try_cancel(resp0 + 16 * sl, respb0 + 8 * sl);
          }
          ++n_req;
        }
        ++nk;
        return true;
      };
      // The remembered chunk holding CTA-local item it (learning chunks as
      // needed): its ordinal, -1 past the last item, -2 when a wait ran out.
      auto locate = [&](int64_t it) -> int {
        while (true) {
          for (int q = nk > kKn ? nk - kKn : 0; q < nk; ++q)
            if (it >= kn[q & (kKn - 1)].lbase && it < kn[q & (kKn - 1)].lbase + kn[q & (kKn - 1)].len) return q;
          if (no_more) return -1;
          if (!learn_next()) return -2;
        }
      };
      int64_t n_fetched = 0;  // own items whose index records were requested (a prefix)
      // The stage record of work item f is f % n_stages, its column tile
      // f / n_stages: followed by cursors on the static schedule (one chunk,
      // items in steps of G), divided out under the dynamic one (whose
      // chunk table already takes the registers).
      ItemCursor fcur, icur;  // the items fetched and the items copied
      auto fetch_idx = [&](int64_t j) -> bool {
        const int q = locate(grp + G * j);
        if (q == -2) return false;
        if (q >= 0) {
          const Chunk &c = kn[q & (kKn - 1)];
          const int64_t fj = c.g0 + (grp + G * j - c.lbase);
          int64_t fs;
          if constexpr (DYN) {
            fs = fj % n_stages;
          } else {
            fcur.to(fj, n_stages);
            fs = fcur.s;
          }
          if (lane == 0) {
            const uint32_t slot = static_cast<uint32_t>(j % kILead);
            const uint8_t *src = pack + fs * kWcsrPackBytes;
            mbar_arrive_expect_tx(ifull_w + 8 * slot, kMetaBytes);
            tma_bulk_load(smem_addr(ring + slot * kMetaBytes), src + kWcsrPackIdxOff, kMetaBytes,
                          ifull_w + 8 * slot);
            if (sub == 0) prefetch_l2_bulk(src + kWcsrPackValOff, kValBytes);
          }
          n_fetched = j + 1;
        }
        return true;
      };
#pragma unroll 1
      for (int j = 0; j < kILead && ok; ++j) ok = fetch_idx(j);
      int64_t consumed = 0;  // own items whose indices were read
      for (int64_t j = 0; ok; ++j) {
        const int64_t it = grp + G * j;
        const int q = locate(it);
        if (q == -2) ok = false;
        if (q < 0) break;
        const Chunk c = kn[q & (kKn - 1)];
        const int64_t f = c.g0 + (it - c.lbase);
        const uint32_t islot = static_cast<uint32_t>(j % kILead);
        ok = mbar_wait_warp(ifull_w + 8 * islot, static_cast<uint32_t>((j / kILead) & 1), p.wait_limit_ns);
        ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
        if (!ok) break;
        const uint8_t *meta = ring + islot * kMetaBytes;
        const int4 d = *reinterpret_cast<const int4 *>(meta + (kWcsrPackDescOff - kWcsrPackIdxOff));
        const int32_t lo = reinterpret_cast<const int32_t *>(meta)[lane];
        const int32_t hi = reinterpret_cast<const int32_t *>(meta)[32 + lane];
        fence_proxy_async_smem();  // these reads before the TMA refill of the slot
        __syncwarp();
        consumed = j + 1;
        ok = fetch_idx(j + kILead);
        if (!ok) break;
        int tile;
        int64_t fsi;
        if constexpr (DYN) {
          tile = static_cast<int>(f / n_stages);
          fsi = f - static_cast<int64_t>(tile) * n_stages;
        } else {
          icur.to(f, n_stages);
          tile = icur.tile;
          fsi = icur.s;
        }
        const uint32_t stage = static_cast<uint32_t>(it % Q);
        const uint32_t phase = static_cast<uint32_t>((it / Q) & 1);
        // the stage is free once the MMAs of item it - Q are complete
        ok = mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns);
        ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
        if (!ok) break;
        const uint32_t st = smem_addr(smem + stage * C_::kStageBytes);
        const uint32_t fb = full0 + 8 * stage;
        if (lane == 0 && sub == 0) {
          if (it == c.lbase) {  // the chunk's partial-sum records (overwritten when used)
            p.partials[2 * c.id] = PartialRec{-1, 0, 0, 0};
            p.partials[2 * c.id + 1] = PartialRec{-1, 0, 0, 0};
          }
          const int32_t fl = d.y | (it == c.lbase ? kRecChunkFirst : 0) | (it == c.lbase + c.len - 1 ? kRecChunkLast : 0);
          stage_rec[stage] = StageRec{d.x, fl, d.z, tile, c.id, {0, 0, 0}};  // released by this arrive
          mbar_arrive_expect_tx(fb, kValBytes);
          tma_bulk_load(st + C_::kGatherBytes, pack + fsi * kWcsrPackBytes + kWcsrPackValOff, kValBytes,
                        fb);
        }
        gather(st, tile * C_::kBN, d.x, lo, hi);
        cp_async_arrive_noinc(fb);
      }
      if (ok && l_end % G == grp) ok = send_end(l_end);
      cp_async_wait_all();
      if (!ok && lane == 0) {
        atomicOr(p.status, kDevTimeout);
        *abort_flag = 1;
        // let the index records and launch-control answers in flight land
        // before the CTA exits
        for (int64_t i = consumed; i < n_fetched; ++i)
          mbar_wait(ifull_w + 8 * (i % kILead), static_cast<uint32_t>((i / kILead) & 1), 1000000ull);
        for (int64_t r = n_read; r < n_req; ++r)
          mbar_wait(respb0 + 8 * (r % kRespSlots), static_cast<uint32_t>((r / kRespSlots) & 1), 1000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp takes the waits (see mbar_wait_warp) and runs the MMA
    // issue converged, one elected lane issuing each MMA and commit; lane 0
    // writes the records for the epilogue.
    {
      constexpr uint32_t idesc = idesc_f16(IN_BF16, /*a_mn_major=*/true, /*b_mn_major=*/false, 128, kH);
      const bool leader = lane == 0;
      uint32_t stage = 0, phase = 0;
      uint32_t seg = 0;     // window segments started
      uint32_t buf = 0;
      int ksteps_done = 0;  // MMA k-steps issued into the current segment
      int32_t s_flags = 0;
      bool s_at_f0 = false;  // the segment starts at its chunk's first item (partial slot 2 chunk)
      bool ok = true;
      auto open_buffer = [&](uint32_t b, uint32_t use) -> bool {
        const bool r = mbar_wait_warp(acce0 + 8 * b, (use & 1u) ^ 1u, p.wait_limit_ns);
        tc_fence_after_sync();
        return __shfl_sync(0xffffffffu, r && !*abort_flag, 0);
      };
      // Items arrive in CTA order until the end record; a segment (the run of
      // one window's stages in this chunk) starts at a window's first stage
      // or a chunk's first item and ends at a window's last stage or a
      // chunk's last item.
      while (ok) {
        ok = mbar_wait_warp(full0 + 8 * stage, phase, p.wait_limit_ns);
        ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
        if (!ok) break;
        const StageRec rec = stage_rec[stage];
        if (rec.flags & kRecEnd) break;
        const bool seg_first = (rec.flags & (kStageFirst | kRecChunkFirst)) != 0;
        const bool seg_last = (rec.flags & (kStageLast | kRecChunkLast)) != 0;
        if (seg_first) {
          buf = seg % kAccBufs;
          if (!open_buffer(buf, seg / kAccBufs)) {
            ok = false;
            break;
          }
          ksteps_done = 0;
          s_flags = rec.flags & kStageFirst;
          s_at_f0 = (rec.flags & kRecChunkFirst) != 0;
        }
        const int ksteps = rec.ncols / 16;
        {
          fence_proxy_async_smem();  // the stage's cp.async writes -> async-proxy MMA reads
          tc_fence_after_sync();
          const uint32_t gath = smem_addr(smem + stage * C_::kStageBytes);  // MMA operand A (MN-major)
          const uint32_t vals = gath + C_::kGatherBytes;                     // MMA operand B (K-major)
          const int nacc = min(NACC, (p.N - rec.tile * C_::kBN + 127) / 128);
          const uint32_t acc = tmem + buf * C_::kAccCols;
          // Descriptors of k step 0; a step adds a fixed byte offset to the
          // start-address field (smem_desc_add), which stays in range.
          const uint64_t bdesc0 = smem_desc_sw128(vals, 16, 1024);
          const uint64_t adesc0 = smem_desc_sw128(gath, kChunkBytes, 1024);
          if (ksteps == kKC / 16 && nacc == NACC) {
            // a full item (the common case): the MMAs without per-step tests,
            // which measured ~20 % cheaper to issue
            const uint32_t acc_in0 = ksteps_done > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < kKC / 16; ++kk) {
              const uint64_t bdesc = smem_desc_add(bdesc0, kk * 32);
#pragma unroll
              for (int a = 0; a < NACC; ++a)
                umma_f16_elect(acc + a * kH, smem_desc_add(adesc0, a * 2 * kChunkBytes + kk * 2048), bdesc, idesc,
                         kk > 0 ? 1u : acc_in0);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < kKC / 16; ++kk) {
              if (kk < ksteps) {
                const uint64_t bdesc = smem_desc_add(bdesc0, kk * 32);
#pragma unroll
                for (int a = 0; a < NACC; ++a) {
                  if (a < nacc)
                    umma_f16_elect(acc + a * kH, smem_desc_add(adesc0, a * 2 * kChunkBytes + kk * 2048), bdesc, idesc,
                             (ksteps_done + kk) > 0 ? 1u : 0u);
                }
              }
            }
          }
          umma_commit_elect(empty0 + 8 * stage);
        }
        ksteps_done += ksteps;
        if (seg_last) {
          s_flags |= rec.flags & kStageLast;
          if (leader) {
            volatile SegRec &sr = seg_rec[buf];
            sr.window = rec.window;
            sr.tile = rec.tile;
            sr.flags = s_flags;
            sr.zero = ksteps_done == 0;
            sr.slot = 2 * rec.chunk + (s_at_f0 ? 0 : 1);
            mbar_arrive(accf0 + 8 * buf);  // releases the record
            umma_commit(accf0 + 8 * buf);  // arrives when the MMAs are done
          }
          ++seg;
        }
        __syncwarp();
        if (++stage == Q) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        // end marker for the epilogue
        buf = seg % kAccBufs;
        ok = open_buffer(buf, seg / kAccBufs);
        if (ok && leader) {
          seg_rec[buf].window = -1;
          mbar_arrive(accf0 + 8 * buf);
          mbar_arrive(accf0 + 8 * buf);
        }
      }
      if (!ok) {
        if (leader) {
          atomicOr(p.status, kDevTimeout);
          *abort_flag = 1;
          umma_commit(drain_bar);
        }
        mbar_wait_warp(drain_bar, 0, 1000000ull);
      }
    }
    __syncwarp();
    grid_launch_dependents();  // every MMA is issued: the reduce pass may be scheduled
  } else {
    // ------------------------------------------------------------ epilogue
    const int sp = warp & 3;
    for (uint32_t seg = 0;; ++seg) {
      const uint32_t buf = seg % kAccBufs;
      const uint32_t use = seg / kAccBufs;
      bool ok = true;
      ok = mbar_wait_warp(accf0 + 8 * buf, use & 1u, p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
      if (!ok) {
        if (lane == 0) {
          atomicOr(p.status, kDevTimeout);
          *abort_flag = 1;
        }
        break;
      }
      const int32_t s_window = seg_rec[buf].window;
      if (s_window < 0) break;
      const int32_t s_tile = seg_rec[buf].tile;
      const int32_t s_flags = seg_rec[buf].flags;
      const bool s_zero = seg_rec[buf].zero != 0;
      const int slot = seg_rec[buf].slot;
      tc_fence_after_sync();
      const bool complete = s_flags == (kStageFirst | kStageLast);
      const int n0 = s_tile * C_::kBN;
      const int nacc = min(NACC, (p.N - n0 + 127) / 128);
      float *ws = p.workspace + static_cast<int64_t>(slot) * kWcsrSlotFloats;
      const int row0 = s_window * kH;
      for (int a = 0; a < nacc; ++a) {
        uint32_t v[16];
        if (!s_zero) {
          tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(sp * 32) << 16) + buf * C_::kAccCols + a * kH, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = 0u;
        }
        const int col = a * 128 + sp * 32 + lane;  // column within the tile
        const int n = n0 + col;
        if (n < p.N) {
          if (complete) {
#pragma unroll
            for (int q = 0; q < kH; ++q)
              if (row0 + q < p.M)
                store_out<OUT_BF16>(p.C, static_cast<int64_t>(row0 + q) * p.N + n, __uint_as_float(v[q]));
          } else {
#pragma unroll
            for (int q = 0; q < kH; ++q) ws[q * 256 + col] = __uint_as_float(v[q]);
          }
        }
      }
      if (!complete && threadIdx.x == 32 * (kMmaWarp + 1))
        p.partials[slot] = PartialRec{s_window, s_tile, s_flags, 0};
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * buf);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C_::kTmemCols);
  }
}

template <int NACC, int Q, int PW, int WPG, int MINB, bool IN_BF16, bool OUT_BF16>
cudaError_t launch_variant(const WcsrParams &p, cudaStream_t stream) {
  using C_ = Cfg<NACC, Q, PW, WPG, MINB, kIdxLead>;
  auto kern = p.dynamic ? wcsr_spmm_kernel<NACC, Q, PW, WPG, MINB, IN_BF16, OUT_BF16, false, true>
                        : wcsr_spmm_kernel<NACC, Q, PW, WPG, MINB, IN_BF16, OUT_BF16, false, false>;
  static std::atomic<uint64_t> smem_set[2];  // per instantiation, one bit per device
  cudaError_t e = set_smem_limit_once(kern, C_::kSmemBytes, smem_set[p.dynamic ? 1 : 0]);
  if (e != cudaSuccess) return e;
  kern<<<p.grid, C_::kThreads, C_::kSmemBytes, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_split_reduce<kH, OUT_BF16>(p.partials, p.workspace, kWcsrSlotFloats, 256, p.C, p.M, p.N, p.grid,
                                           C_::kBN, stream);
}

template <int NACC, int Q, int PW, int WPG, int MINB>
cudaError_t launch_dtypes(const WcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t s) {
  if (in_bf16)
    return out_bf16 ? launch_variant<NACC, Q, PW, WPG, MINB, true, true>(p, s)
                    : launch_variant<NACC, Q, PW, WPG, MINB, true, false>(p, s);
  return out_bf16 ? launch_variant<NACC, Q, PW, WPG, MINB, false, true>(p, s)
                  : launch_variant<NACC, Q, PW, WPG, MINB, false, false>(p, s);
}

// ------------------------------------------------------------ no-allocation variant
// Builds the stage list of spmm_wcsr_run_noalloc on the device: one block,
// each thread walks a contiguous run of windows, counts their stages
// (ceil(P_w / 64), at least 1), a block-wide exclusive scan places the runs,
// and the threads write their stages.  The total goes to *n_stages.
//
// The caller's window_row_ptr is checked first, since the host cannot read
// it: window_row_ptr[0] == 0, entries non-decreasing and multiples of 16 (the
// value copies are 16-byte cp.async and the MMA takes 16 columns per step),
// window_row_ptr[n_windows] == p_total, and the stage count within the
// scratch's stage area.  On any failure no stage is written, *n_stages is 0
// (the product kernel then does no work and C is left as it was) and
// kDevIndex is set in the scratch's status word.
__global__ void __launch_bounds__(1024)
    wcsr_noalloc_stages_kernel(const int64_t *window_row_ptr, int64_t n_windows, int64_t p_total,
                               WcsrStage *stages, int64_t *n_stages, uint32_t *status) {
  __shared__ int64_t part[1024];
  const int t = threadIdx.x;
  if (t == 0) *status = 0;  // the scratch keeps the previous call's contents
  const int64_t per = (n_windows + blockDim.x - 1) / blockDim.x;
  const int64_t w0 = t * per < n_windows ? t * per : n_windows;
  const int64_t w1 = w0 + per < n_windows ? w0 + per : n_windows;
  int64_t cnt = 0;
  bool bad = (t == 0 && window_row_ptr[0] != 0) || (t == 1023 && window_row_ptr[n_windows] != p_total);
  for (int64_t w = w0; w < w1 && !bad; ++w) {
    const int64_t b = window_row_ptr[w], e = window_row_ptr[w + 1];
    if (e < b || (e & 15) != 0) {
      bad = true;
      break;
    }
    const int64_t pw = e - b;
    cnt += pw > 0 ? (pw + kKC - 1) / kKC : 1;
  }
  part[t] = cnt;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan (Hillis-Steele)
    const int64_t v = t >= off ? part[t - off] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  // every thread sees the same total; a bad entry anywhere rejects the call
  if (__syncthreads_or(bad ? 1 : 0) || part[1023] > kNoallocMaxStages) {
    if (t == 0) {
      *n_stages = 0;
      *status = kDevIndex;
    }
    return;
  }
  int64_t pos = part[t] - cnt;
  for (int64_t w = w0; w < w1; ++w) {
    const int64_t b = window_row_ptr[w], e = window_row_ptr[w + 1];
    if (e == b) {
      stages[pos++] = WcsrStage{static_cast<int32_t>(b), static_cast<int32_t>(w), 0, kStageFirst | kStageLast};
      continue;
    }
    for (int64_t q = b; q < e; q += kKC) {
      const int32_t flags = (q == b ? kStageFirst : 0) | (q + kKC >= e ? kStageLast : 0);
      stages[pos++] = WcsrStage{static_cast<int32_t>(q), static_cast<int32_t>(w),
                                static_cast<int32_t>(e - q < kKC ? e - q : kKC), flags};
    }
  }
  if (t == 1023) *n_stages = part[1023];
}

template <int NACC, int Q, bool IN_BF16, bool OUT_BF16>
cudaError_t launch_noalloc_variant(const WcsrParams &p, cudaStream_t stream) {
  using C_ = Cfg<NACC, Q, 4, 1, 1, 0>;
  auto kern = wcsr_spmm_kernel<NACC, Q, 4, 1, 1, IN_BF16, OUT_BF16, true>;
  static std::atomic<uint64_t> smem_set{0};  // per instantiation, one bit per device
  cudaError_t e = set_smem_limit_once(kern, C_::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  kern<<<p.grid, C_::kThreads, C_::kSmemBytes, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_split_reduce<kH, OUT_BF16>(p.partials, p.workspace, kWcsrSlotFloats, 256, p.C, p.M, p.N, p.grid,
                                           C_::kBN, stream);
}

// Scratch of spmm_wcsr_run_noalloc: stage list, partial-sum slots (two per
// CTA), partial records and the stage count.  Held by every GPU that loads
// the library, for the life of the process.
constexpr size_t kNoallocStageBytes = static_cast<size_t>(kNoallocMaxStages) * sizeof(WcsrStage);
constexpr size_t kNoallocWsBytes = static_cast<size_t>(2 * kNoallocMaxCtas) * kWcsrSlotFloats * sizeof(float);
constexpr size_t kNoallocRecBytes = static_cast<size_t>(2 * kNoallocMaxCtas) * sizeof(PartialRec);
constexpr size_t kNoallocScratchBytes = kNoallocStageBytes + kNoallocWsBytes + kNoallocRecBytes + 256;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

}  // namespace

size_t wcsr_noalloc_scratch_bytes() { return kNoallocScratchBytes; }

namespace {
// Device address of the scratch array on the current device, looked up once
// per device with that device current (in host code the array's name is only
// a stand-in).
cudaError_t noalloc_base(uint8_t **base) {
  static std::mutex mu;
  static uint8_t *addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<uint8_t *>(ptr);
  }
  *base = addr[dev];
  return cudaSuccess;
}

// The status word (bounded-wait timeouts, the stage-list check) in the
// scratch's spare tail.
constexpr size_t kNoallocStatusOff = kNoallocStageBytes + kNoallocWsBytes + kNoallocRecBytes + 8;
}  // namespace

cudaError_t wcsr_noalloc_take_status(uint32_t *word, cudaStream_t stream) {
  uint8_t *base = nullptr;
  cudaError_t e = noalloc_base(&base);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(word, base + kNoallocStatusOff, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(base + kNoallocStatusOff, 0, sizeof(uint32_t), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

cudaError_t launch_wcsr_noalloc(WcsrParams p, const int64_t *window_row_ptr, int64_t n_windows, int num_sms,
                                bool in_bf16, bool out_bf16, cudaStream_t stream) {
  uint8_t *base = nullptr;
  cudaError_t e = noalloc_base(&base);
  if (e != cudaSuccess) return e;
  WcsrStage *stages = reinterpret_cast<WcsrStage *>(base);
  p.stages = stages;
  p.workspace = reinterpret_cast<float *>(base + kNoallocStageBytes);
  p.partials = reinterpret_cast<PartialRec *>(base + kNoallocStageBytes + kNoallocWsBytes);
  uint8_t *tail = base + kNoallocStageBytes + kNoallocWsBytes + kNoallocRecBytes;  // 256 spare bytes
  p.n_stages_dev = reinterpret_cast<int64_t *>(tail);
  p.status = reinterpret_cast<uint32_t *>(base + kNoallocStatusOff);  // read by wcsr_noalloc_take_status
  p.grid = num_sms < kNoallocMaxCtas ? num_sms : kNoallocMaxCtas;
  p.dynamic = 0;
  wcsr_noalloc_stages_kernel<<<1, 1024, 0, stream>>>(window_row_ptr, n_windows, p.P_total, stages,
                                                      reinterpret_cast<int64_t *>(tail), p.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.N <= 128) {
    if (in_bf16) return out_bf16 ? launch_noalloc_variant<1, 10, true, true>(p, stream)
                                 : launch_noalloc_variant<1, 10, true, false>(p, stream);
    return out_bf16 ? launch_noalloc_variant<1, 10, false, true>(p, stream)
                    : launch_noalloc_variant<1, 10, false, false>(p, stream);
  }
  if (in_bf16) return out_bf16 ? launch_noalloc_variant<2, 5, true, true>(p, stream)
                               : launch_noalloc_variant<2, 5, true, false>(p, stream);
  return out_bf16 ? launch_noalloc_variant<2, 5, false, true>(p, stream)
                  : launch_noalloc_variant<2, 5, false, false>(p, stream);
}

// Two CTAs per SM at every N (see launch_wcsr for their shapes): one CTA's
// barrier handshakes and MMA issue stalls overlap the other's work.
int wcsr_ctas_per_sm(int64_t N) {
  (void)N;
  return 2;
}

// Whether N > 128 takes 256-column work items (one gather of a full B row
// per stage) instead of 128-column ones.
constexpr bool kWideTiles = true;

int wcsr_tile_cols(int64_t N) { return (N <= 128 || !kWideTiles) ? 128 : 256; }

// Launch shapes, two CTAs per SM (one CTA per SM with more stages and
// producers measured 35-70 % slower: the single MMA-issuing thread of a CTA
// becomes the limit).  128-column items: five 18 KB stages, five producer
// warps each copying whole items (7-10 % faster than four; eight warps in
// groups of two were slower).  256-column items: three 34 KB stages, three
// producer groups of two warps (each warp copies 32 of an item's 64 rows):
// 12 copying warps per SM instead of 6, 7 % faster on the uniform matrix.
cudaError_t launch_wcsr(const WcsrParams &p, bool in_bf16, bool out_bf16, cudaStream_t stream) {
  if (p.n_stages == 0 || p.N == 0 || p.grid == 0) return cudaSuccess;
  if (wcsr_tile_cols(p.N) == 128) return launch_dtypes<1, 5, 5, 1, 2>(p, in_bf16, out_bf16, stream);
  return launch_dtypes<2, 3, 6, 2, 2>(p, in_bf16, out_bf16, stream);
}

}  // namespace spmm
