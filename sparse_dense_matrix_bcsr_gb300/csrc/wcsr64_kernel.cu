// wcsr64_kernel.cu -- WCSR SpMM with 64-row windows for sm_103a.
//
// Method: "AsyncSparse", Section II-C (WCSR) with the window height the paper
// evaluates WCSR at (Section IV-A: windows of 64 rows, column padding 8),
// Section III-B (a window's packed value tile is contiguous; the rows of B it
// multiplies are gathered through window_col_idx by all threads, written to
// shared memory with the 128-byte swizzle applied by hand) and Section III-C
// (long windows split between CTAs).  The paper runs this configuration in
// TF32; here the values and B are 16-bit (bf16 / fp16) with fp32
// accumulation, the kind the gathered rows can feed the tensor cores in as
// they lie (dense columns contiguous).
//
// A 64-row window makes the product the same shape as a BCSR block row: a
// stage is 64 packed columns of one window, its 64 x 64 value tile is the
// MMA's M = 64 operand (K-major, pre-swizzled in the stage record) and the 64
// gathered rows of B, 256 columns wide, its N = 256 operand (MN-major), one
// weight-stationary M = 64 x N = 256 x K = 16 MMA per k step into an
// accumulator of 128 TMEM columns (rows 0..63 in lanes 0..63 for columns
// 0..127, in lanes 64..127 for columns 128..255).
//
// Work list and split: as in wcsr_kernel.cu -- the T = stages x column tiles
// work items are cut into equal contiguous shares, one per persistent CTA; a
// CTA's run of stages of one window is a segment; a segment holding the whole
// window is stored to C through TMA stores, a cut one is written as fp32
// partial sums (64 x 256) for split_reduce_kernel.
//
// PW + 5 warps (see kLaunch* for the launch shape):
//   warps 0..PW-1  producers in groups of WPG: group g owns the work items
//                  g, g + PW/WPG, ...; each warp of the group gathers its
//                  share of an item's 64 rows of B with 16-byte cp.async (one
//                  512-byte row per instruction at full width, live columns
//                  only when N is narrower), after fetching the index record
//                  ahead into a per-warp ring; the group's first warp has the
//                  value tile copied into the stage (TMA bulk copy)
//   warp PW        TMEM allocator and MMA issuer
//   warps PW+1..   epilogue (warp w reads TMEM sub-partition w % 4)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "split_reduce.cuh"

namespace spmm {
namespace {

constexpr int kH = 64;
constexpr int kKC = 64;                                // packed columns per stage
constexpr int kValBytes = kH * kKC * 2;                // 8 KB value tile
constexpr int kIdxOff = wcsr_pack_idx_off(kH);
constexpr int kMetaBytes = wcsr_pack_bytes(kH) - kIdxOff;  // indices + descriptor
constexpr int kPackBytes = wcsr_pack_bytes(kH);
constexpr int kBN = 256;                               // columns of C per tile
constexpr int kChunkBytes = kKC * 128;                 // 64 gathered rows x 64 columns
constexpr int kGatherBytes = 4 * kChunkBytes;          // 32 KB
constexpr int kStageBytes = kValBytes + kGatherBytes;  // 40 KB
constexpr int kEpiWarps = 4;
constexpr int kAccCols = kBN / 2;
constexpr int kNbuf = 2;
constexpr int kTmemCols = kNbuf * kAccCols;
constexpr int kBoxBytes = 2048;                         // a store box: 32 rows x 64 bytes
constexpr int kMiscBytes = 1024;

// Q stages, PW producer warps in groups of WPG (the warps of a group copy
// disjoint row ranges of the same items: a warp's cp.async issue rate is
// limited, so more copying warps gather faster), MINB CTAs per SM.  Each
// producer warp fetches its items' index records kILead of its items ahead.
template <int Q, int PW, int WPG, int MINB, bool OUT_BF16>
struct Cfg {
  static constexpr int kQ = Q;
  static constexpr int kPW = PW;
  static constexpr int kG = PW / WPG;                   // producer groups
  static constexpr int kILead = WPG > 1 ? 2 : 4;
  static constexpr int kMmaWarp = PW;
  static constexpr int kEpiWarp0 = PW + 1;
  static constexpr int kThreads = 32 * (PW + 1 + kEpiWarps);
  static constexpr int kOutBytes = OUT_BF16 ? 2 : 4;
  static constexpr int kBoxCols = 64 / kOutBytes;       // C columns per box
  static constexpr int kParts = OUT_BF16 ? 4 : 8;       // the warp's 128 columns in parts of one box
  static constexpr int kPartCols = 128 / kParts;
  static constexpr int kStaging = kEpiWarps * 2 * kBoxBytes;
  static constexpr int kIdxRingBytes = (PW * kILead * kMetaBytes + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = Q * kStageBytes + kStaging + kIdxRingBytes + kMiscBytes + 1024;
  static_assert(kPartCols == kBoxCols, "one store box per part");
  static_assert(kSmemBytes <= 227 * 1024 && MINB * (kSmemBytes + 1024) <= 228 * 1024, "shared memory");
  static_assert(MINB * kTmemCols <= 512, "TMEM");
  // a warp waits for its item's stage with a parity wait on the MMA commit of
  // item it - Q; unambiguous only if the commit of it - 2Q was already seen,
  // which the warp's previous wait (item it - kG) guarantees when kG <= Q
  static_assert(PW % WPG == 0 && (WPG == 1 || WPG == 2), "producer groups");
  static_assert(kG <= Q, "more producer groups than stages");
};

struct StageRec {  // producer -> MMA
  int32_t ncols;
  int32_t flags;
  int32_t window;
  int32_t tile;
};
struct SegRec {    // MMA -> epilogue
  int32_t window;  // -1: no more segments
  int32_t tile;
  int32_t flags;   // kStageFirst | kStageLast of the window, as covered by this CTA
  int32_t zero;    // no MMA was issued
  int32_t slot;    // workspace slot of a cut segment
  int32_t pad_[3];
};

template <int Q, int PW, int WPG, int MINB, bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(32 * (PW + 5), MINB)
    wcsr64_spmm_kernel(const __grid_constant__ CUtensorMap tmC, const WcsrParams p) {
  using E = Cfg<Q, PW, WPG, MINB, OUT_BF16>;
  constexpr int kIdxLead = E::kILead;
  constexpr int kQ = E::kQ;
  constexpr int kPW = E::kPW;
  constexpr int kMmaWarp = E::kMmaWarp;
  constexpr int kEpiWarp0 = E::kEpiWarp0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *staging = smem + kQ * kStageBytes;
  uint8_t *iring = staging + E::kStaging;
  uint64_t *bars = reinterpret_cast<uint64_t *>(iring + E::kIdxRingBytes);
  // bars: full[kQ], empty[kQ], acc_full[kNbuf], acc_empty[kNbuf], drain, ifull[kPW][kIdxLead]
  constexpr int kBars = 2 * kQ + 2 * kNbuf + 1 + kPW * kIdxLead;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  StageRec *stage_rec = reinterpret_cast<StageRec *>(tmem_slot + 4);              // [kQ]
  volatile SegRec *seg_rec = reinterpret_cast<volatile SegRec *>(stage_rec + kQ);  // [kNbuf]
  static_assert(kBars * 8 + 16 + kQ * 16 + kNbuf * 32 <= kMiscBytes, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_col_tiles = (p.N + kBN - 1) / kBN;
  const int64_t n_stages = p.n_stages;
  const int64_t total = n_stages * n_col_tiles;
  const int64_t f0 = total * blockIdx.x / gridDim.x;
  const int64_t f1 = total * (blockIdx.x + 1) / gridDim.x;

  const uint32_t full0 = smem_addr(&bars[0]);
  const uint32_t empty0 = smem_addr(&bars[kQ]);
  const uint32_t accf0 = smem_addr(&bars[2 * kQ]);
  const uint32_t acce0 = smem_addr(&bars[2 * kQ + kNbuf]);
  const uint32_t drain_bar = smem_addr(&bars[2 * kQ + 2 * kNbuf]);
  const uint32_t ifull0 = smem_addr(&bars[2 * kQ + 2 * kNbuf + 1]);

  if (threadIdx.x == 0) {
    for (int q = 0; q < kQ; ++q) {
      // 32 cp.async lane arrivals of each warp of the owning group + the
      // group's first warp's lane 0 arrive (stage record, value tile bytes)
      mbar_init(full0 + 8 * q, 1 + 32 * WPG);
      mbar_init(empty0 + 8 * q, 1);
    }
    for (int b = 0; b < kNbuf; ++b) {
      mbar_init(accf0 + 8 * b, 2);
      mbar_init(acce0 + 8 * b, kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int v = 0; v < kPW * kIdxLead; ++v) mbar_init(ifull0 + 8 * v, 1);  // lane 0's expect_tx arrive
    *abort_flag = 0;
    fence_barrier_init();
    p.partials[2 * blockIdx.x] = PartialRec{-1, 0, 0, 0};
    p.partials[2 * blockIdx.x + 1] = PartialRec{-1, 0, 0, 0};
    tma_prefetch_desc(&tmC);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < kPW) {
    // ------------------------------------------------------------ producers
    // Group g (warps g*WPG .. g*WPG+WPG-1) owns the work items g, g + kG, ...
    // of the CTA's share; each of its warps copies rows [rbeg, rend) of them.
    // Each warp
    // fetches the index record of its item j (272 bytes) kIdxLead of its items
    // ahead into slot j % kIdxLead of its ring, reads the item's indices from
    // there, waits for the item's stage to be free, has the value tile copied
    // into the stage by TMA and copies the item's 64 rows of B with cp.async.
    // A warp's gather completes before the warp moves on (the copies of one
    // item are in flight while it issues them), so the stages loading at once
    // are the producer warps' items: PW <= Q keeps them all busy and the
    // parity waits unambiguous.
    const uint16_t *Bp = reinterpret_cast<const uint16_t *>(p.B);
    constexpr int kG = E::kG;
    const int grp = warp / WPG, sub = warp % WPG;
    const int rbeg = sub * (64 / WPG), rend = rbeg + 64 / WPG;
    const uint8_t *pack = reinterpret_cast<const uint8_t *>(p.stage_pack);
    uint8_t *ring = iring + warp * kIdxLead * kMetaBytes;
    const uint32_t ifull_w = ifull0 + 8 * (warp * kIdxLead);
    ItemCursor fcur, icur;  // the items fetched and the items copied
    auto fetch_idx = [&](int64_t j) {
      const int64_t fj = f0 + grp + j * kG;
      if (fj < f1) fcur.to(fj, n_stages);
      if (fj < f1 && lane == 0) {
        const uint32_t slot = static_cast<uint32_t>(j % kIdxLead);
        const uint8_t *src = pack + fcur.s * kPackBytes;
        mbar_arrive_expect_tx(ifull_w + 8 * slot, kMetaBytes);
        tma_bulk_load(smem_addr(ring + slot * kMetaBytes), src + kIdxOff, kMetaBytes, ifull_w + 8 * slot);
        if (sub == 0) prefetch_l2_bulk(src, kValBytes);
      }
    };
    // The item's 64 rows of B -> the stage's gather area: one B row per
    // instruction when all 32 units of 16 bytes are live, else live units
    // only, several rows per instruction; a padding position (-1) is
    // zero-filled.  lo / hi hold the indices of rows lane and 32 + lane.
    auto gather = [&](uint32_t st, int n0, int ncols, int32_t lo, int32_t hi) {
      const int live_units = (min(kBN, p.N - n0) + 7) >> 3;  // 1 .. 32
      const int rlim = min(ncols, rend);
      const uint32_t dst = st + kValBytes;
      if (live_units == 32) {
        const int n = n0 + lane * 8;
        const uint32_t dst_col = (lane >> 3) * kChunkBytes;
        const uint32_t uu = static_cast<uint32_t>(lane & 7);
        for (int r0 = rbeg; r0 < rlim; r0 += 16) {
          const int32_t src = r0 < 32 ? lo : hi;
          int32_t col[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) col[j] = __shfl_sync(0xffffffffu, src, (r0 + j) & 31);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = r0 + j;
            const bool live = col[j] >= 0;
            cp_async_16(dst + dst_col + r * 128 + ((uu ^ static_cast<uint32_t>(r & 7)) << 4),
                        live ? static_cast<const void *>(Bp + static_cast<int64_t>(col[j]) * p.N + n)
                             : static_cast<const void *>(Bp),
                        live ? 16u : 0u);
          }
        }
        return;
      }
      const int sh = 32 - __clz(live_units - 1);
      const int rsh = 5 - sh;
      const int i_beg = rbeg >> rsh;  // instructions holding rows [rbeg, rlim)
      const int i_end = (rlim + (1 << rsh) - 1) >> rsh;
      const int r_lane = lane >> sh;
      const int u = lane & ((1 << sh) - 1);
      const int n = n0 + u * 8;
      const bool u_live = n < p.N;
      const uint32_t dst_u = (u >> 3) * kChunkBytes;
      const uint32_t uu = static_cast<uint32_t>(u & 7);
      for (int i0 = i_beg; i0 < i_end; i0 += 16) {
        int32_t col[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int rb = (i0 + j) << rsh;
          col[j] = __shfl_sync(0xffffffffu, rb < 32 ? lo : hi, (rb + r_lane) & 31);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = ((i0 + j) << rsh) + r_lane;
          if (i0 + j < i_end && u_live && r >= rbeg && r < rlim) {
            const bool live = col[j] >= 0;
            cp_async_16(dst + dst_u + r * 128 + ((uu ^ static_cast<uint32_t>(r & 7)) << 4),
                        live ? static_cast<const void *>(Bp + static_cast<int64_t>(col[j]) * p.N + n)
                             : static_cast<const void *>(Bp),
                        live ? 16u : 0u);
          }
        }
      }
    };
#pragma unroll 1
    for (int j = 0; j < kIdxLead; ++j) fetch_idx(j);
    bool ok = true;
    int64_t consumed = 0;  // own items whose indices were read; fetches of the next kIdxLead are in flight
    for (int64_t j = 0;; ++j) {
      const int64_t f = f0 + grp + j * kG;
      if (f >= f1) break;
      const uint32_t islot = static_cast<uint32_t>(j % kIdxLead);
      ok = mbar_wait_warp(ifull_w + 8 * islot, static_cast<uint32_t>((j / kIdxLead) & 1), p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
      if (!ok) break;
      const uint8_t *meta = ring + islot * kMetaBytes;
      const int4 d = *reinterpret_cast<const int4 *>(meta + 256);  // {ncols, flags, window, 0}
      const int32_t lo = reinterpret_cast<const int32_t *>(meta)[lane];
      const int32_t hi = reinterpret_cast<const int32_t *>(meta)[32 + lane];
      fence_proxy_async_smem();  // these reads before the TMA refill of the slot
      __syncwarp();
      fetch_idx(j + kIdxLead);
      consumed = j + 1;
      icur.to(f, n_stages);
      const int tile = icur.tile;
      const int64_t it = f - f0;
      const uint32_t stage = static_cast<uint32_t>(it % kQ);
      const uint32_t phase = static_cast<uint32_t>((it / kQ) & 1);
      ok = mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
      if (!ok) break;
      const uint32_t st = smem_addr(smem + stage * kStageBytes);
      const uint32_t fb = full0 + 8 * stage;
      if (lane == 0 && sub == 0) {
        stage_rec[stage] = StageRec{d.x, d.y, d.z, tile};  // released by this arrive
        mbar_arrive_expect_tx(fb, kValBytes);
        tma_bulk_load(st, pack + icur.s * kPackBytes, kValBytes, fb);
      }
      gather(st, tile * kBN, d.x, lo, hi);
      cp_async_arrive_noinc(fb);
    }
    cp_async_wait_all();
    if (!ok && lane == 0) {
      atomicOr(p.status, kDevTimeout);
      *abort_flag = 1;
      for (int64_t i = consumed; i < consumed + kIdxLead && f0 + grp + i * kG < f1; ++i)
        mbar_wait(ifull_w + 8 * (i % kIdxLead), static_cast<uint32_t>((i / kIdxLead) & 1), 1000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_f16(IN_BF16, /*a_mn_major=*/false, /*b_mn_major=*/true, 64, kBN);
    const bool leader = lane == 0;
    uint32_t stage = 0, phase = 0, seg = 0, buf = 0;
    int ksteps_done = 0;
    int32_t s_flags = 0;
    bool s_at_f0 = false;
    bool ok = true;
    auto open_buffer = [&](uint32_t b, uint32_t use) -> bool {
      const bool r = mbar_wait_warp(acce0 + 8 * b, (use & 1u) ^ 1u, p.wait_limit_ns);
      tc_fence_after_sync();
      return __shfl_sync(0xffffffffu, r && !*abort_flag, 0);
    };
    for (int64_t f = f0; f < f1 && ok; ++f) {
      ok = mbar_wait_warp(full0 + 8 * stage, phase, p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok && !*abort_flag, 0);
      if (!ok) break;
      const StageRec rec = stage_rec[stage];
      const bool seg_first = f == f0 || (rec.flags & kStageFirst);
      const bool seg_last = f == f1 - 1 || (rec.flags & kStageLast);
      if (seg_first) {
        buf = seg % kNbuf;
        if (!open_buffer(buf, seg / kNbuf)) {
          ok = false;
          break;
        }
        ksteps_done = 0;
        s_flags = rec.flags & kStageFirst;
        s_at_f0 = f == f0;
      }
      const int ksteps = rec.ncols / 16;
      {  // converged: one elected lane issues each MMA and commit
        fence_proxy_async_smem();  // the stage's cp.async writes -> async-proxy MMA reads
        tc_fence_after_sync();
        const uint32_t vals = smem_addr(smem + stage * kStageBytes);  // M operand (K-major)
        const uint32_t gath = vals + kValBytes;                       // N operand (MN-major)
        const uint32_t acc = tmem + buf * kAccCols;
        const uint64_t vdesc0 = smem_desc_sw128(vals, 16, 1024);
        const uint64_t gdesc0 = smem_desc_sw128(gath, kChunkBytes, 1024);
        if (ksteps == kKC / 16) {  // a full item: no per-step tests (cheaper to issue)
          const uint32_t acc_in0 = ksteps_done > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < kKC / 16; ++kk)
            umma_ws_f16_elect(acc, smem_desc_add(vdesc0, kk * 32), smem_desc_add(gdesc0, kk * 2048), idesc,
                        kk > 0 ? 1u : acc_in0);
        } else {
#pragma unroll
          for (int kk = 0; kk < kKC / 16; ++kk)
            if (kk < ksteps)
              umma_ws_f16_elect(acc, smem_desc_add(vdesc0, kk * 32), smem_desc_add(gdesc0, kk * 2048), idesc,
                          (ksteps_done + kk) > 0 ? 1u : 0u);
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
          sr.slot = 2 * static_cast<int32_t>(blockIdx.x) + (s_at_f0 ? 0 : 1);
          mbar_arrive(accf0 + 8 * buf);
          umma_commit(accf0 + 8 * buf);
        }
        ++seg;
      }
      __syncwarp();
      if (++stage == kQ) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (ok) {
      buf = seg % kNbuf;
      ok = open_buffer(buf, seg / kNbuf);
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
      if (leader)
        for (int b = 0; b < kNbuf; ++b) {
          mbar_arrive(accf0 + 8 * b);
          mbar_arrive(accf0 + 8 * b);
        }
    }
    grid_launch_dependents();  // every MMA is issued: the reduce pass may be scheduled
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads sub-partition sp = w % 4: rows 32 (sp % 2) + lane of the
    // window, columns 128 (sp / 2) .. + 127 of the tile.  A whole window goes
    // to C through the warp's staging area (32-row x 64-byte boxes, 64-byte
    // swizzle, two buffers alternating) and TMA stores; a cut one goes to its
    // fp32 workspace slot with plain stores.
    const int sp = warp & 3;
    uint8_t *stg = staging + (warp - kEpiWarp0) * 2 * kBoxBytes;
    const uint32_t row_sw = static_cast<uint32_t>((lane >> 1) & 3);
    uint32_t pcount = 0;
    for (uint32_t seg = 0;; ++seg) {
      const uint32_t buf = seg % kNbuf;
      const bool r = mbar_wait_warp(accf0 + 8 * buf, (seg / kNbuf) & 1u, p.wait_limit_ns);
      if (!__shfl_sync(0xffffffffu, r && !*abort_flag, 0)) {
        if (lane == 0 && !r) {
          atomicOr(p.status, kDevTimeout);
          *abort_flag = 1;
        }
        break;
      }
      const int32_t s_window = seg_rec[buf].window;
      if (s_window < 0) break;
      const int32_t s_tile = seg_rec[buf].tile;
      const int32_t s_flags = seg_rec[buf].flags;
      const bool zero = seg_rec[buf].zero != 0;
      const int slot = seg_rec[buf].slot;
      tc_fence_after_sync();
      const bool complete = s_flags == (kStageFirst | kStageLast);
      const int rloc = (sp & 1) * 32;                 // first row of this warp within the window
      const int row0 = s_window * kH + rloc;
      const int c0 = (sp >> 1) * 128;                 // first column of this warp within the tile
      const int n0 = s_tile * kBN + c0;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(sp * 32) << 16) + buf * kAccCols;
      if (complete) {
#pragma unroll 1
        for (int part = 0; part < E::kParts; ++part) {
          uint8_t *pst = stg + (pcount & 1) * kBoxBytes;
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
          uint32_t v[E::kPartCols / 16][16];
#pragma unroll
          for (int g = 0; g < E::kPartCols / 16; ++g) {
            if (!zero) {
              tmem_ld_32x32b_x16(tbase + part * E::kPartCols + g * 16, v[g]);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) v[g][i] = 0u;
            }
          }
          if (!zero) tmem_ld_wait();
          uint8_t *row = pst + lane * 64;
#pragma unroll
          for (int g = 0; g < E::kPartCols / 16; ++g) {
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
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4 *>(row + ((static_cast<uint32_t>(q) ^ row_sw) << 4)) =
                    make_uint4(v[g][4 * q], v[g][4 * q + 1], v[g][4 * q + 2], v[g][4 * q + 3]);
            }
          }
          if (part == E::kParts - 1) tc_fence_before_sync();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (part == E::kParts - 1) mbar_arrive(acce0 + 8 * buf);
            const int x = n0 + part * E::kPartCols;
            if (row0 < p.M && x < p.N) tma_store_2d(&tmC, smem_addr(pst), x, row0);
            bulk_commit_group();
          }
          ++pcount;
        }
      } else {
        float *ws = p.workspace + static_cast<int64_t>(slot) * kWcsr64SlotFloats;
#pragma unroll 1
        for (int g = 0; g < 128 / 16; ++g) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tbase + g * 16, v);
          tmem_ld_wait();
          if (s_tile * kBN + c0 + g * 16 < p.N) {
            float4 *dst = reinterpret_cast<float4 *>(ws + (rloc + lane) * kBN + c0 + g * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if (warp == kEpiWarp0) p.partials[slot] = PartialRec{s_window, s_tile, s_flags, 0};
          mbar_arrive(acce0 + 8 * buf);
        }
      }
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

template <int Q, int PW, int WPG, int MINB, bool IN_BF16, bool OUT_BF16>
cudaError_t launch_variant(const CUtensorMap &tmC, const WcsrParams &p, cudaStream_t stream) {
  using E = Cfg<Q, PW, WPG, MINB, OUT_BF16>;
  auto kern = wcsr64_spmm_kernel<Q, PW, WPG, MINB, IN_BF16, OUT_BF16>;
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_smem_limit_once(kern, E::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  kern<<<p.grid, E::kThreads, E::kSmemBytes, stream>>>(tmC, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_split_reduce<kH, OUT_BF16>(p.partials, p.workspace, kWcsr64SlotFloats, kBN, p.C, p.M, p.N, p.grid,
                                           kBN, stream);
}

}  // namespace

// Launch shape: kLaunchQ stages, kLaunchPW producer warps in groups of
// kLaunchWPG, kLaunchMinB CTAs per SM.
constexpr int kLaunchQ = 5, kLaunchPW = 10, kLaunchWPG = 2, kLaunchMinB = 1;

int wcsr64_ctas_per_sm() { return kLaunchMinB; }

cudaError_t launch_wcsr64(const CUtensorMap &tmC, const WcsrParams &p, bool in_bf16, bool out_bf16,
                          cudaStream_t stream) {
  if (p.n_stages == 0 || p.N == 0 || p.grid == 0) return cudaSuccess;
  constexpr int Q = kLaunchQ, PW = kLaunchPW, G = kLaunchWPG, MB = kLaunchMinB;
  if (in_bf16)
    return out_bf16 ? launch_variant<Q, PW, G, MB, true, true>(tmC, p, stream)
                    : launch_variant<Q, PW, G, MB, true, false>(tmC, p, stream);
  return out_bf16 ? launch_variant<Q, PW, G, MB, false, true>(tmC, p, stream)
                  : launch_variant<Q, PW, G, MB, false, false>(tmC, p, stream);
}

}  // namespace spmm
