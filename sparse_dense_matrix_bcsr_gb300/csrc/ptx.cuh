// ptx.cuh -- inline-PTX building blocks for sm_103a: mbarriers with bounded
// waits, TMA tile loads, tcgen05 (TMEM allocation, MMA, commit, loads) and the
// shared-memory matrix descriptors the MMA reads its operands through.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace spmm {

// Bits of the per-handle device status word.
constexpr uint32_t kDevTimeout = 1u;
constexpr uint32_t kDevIndex = 2u;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One probe of the phase: true once the phase with this parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait until the phase with the given parity has completed, for at most
// limit_ns nanoseconds.  Returns false when the limit ran out; no wait in
// this library is unbounded.  After two quick probes the thread sleeps
// between probes (32 ns doubling to 256 ns): on GB300 a warp polling an
// mbarrier in a tight loop occupies the shared-memory pipe that the copying
// warps' cp.async needs (four polling warps cut a gather pipeline's rate to a
// third).  The bound is counted with the SM's cycle counter at 2.1 GHz, so at
// lower clocks the wait lasts proportionally longer but still ends.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity) || mbar_try_wait(bar, parity)) return true;
  const long long limit_cycles = static_cast<long long>(limit_ns) * 21 / 10;
  const long long t0 = clock64();
  uint32_t sleep_ns = 32;
  while (true) {
    __nanosleep(sleep_ns);
    if (sleep_ns < 256) sleep_ns <<= 1;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit_cycles) return false;
  }
}

// The same wait taken by a whole converged warp: every lane probes, lane 0's
// result decides for all.  Measured on GB300: a gather pipeline whose warps
// waited with lane 0 alone (the other lanes parked at a warp barrier) ran at a
// third of the rate it reached when all 32 lanes took the wait together, so
// every role in this library that has whole warps waits this way.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (__shfl_sync(0xffffffffu, mbar_try_wait(bar, parity) ? 1 : 0, 0)) return true;
  const long long limit_cycles = static_cast<long long>(limit_ns) * 21 / 10;
  const long long t0 = clock64();
  uint32_t sleep_ns = 32;
  while (true) {
    __nanosleep(sleep_ns);
    if (sleep_ns < 128) sleep_ns <<= 1;
    int state = mbar_try_wait(bar, parity) ? 1 : (clock64() - t0 > limit_cycles ? 2 : 0);
    state = __shfl_sync(0xffffffffu, state, 0);
    if (state != 0) return state == 1;
  }
}

// ---------------------------------------------------------------- dependent launches
// A kernel launched with programmatic stream serialization may start before
// the kernel ahead of it in the stream has finished: it waits here until that
// kernel has completed and its memory writes are visible (a no-op for a
// kernel launched without the attribute).  The kernel ahead lets its
// dependents be scheduled once every one of its CTAs has executed
// launch_dependents or exited.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// umma_f16 / umma_commit issued by a whole converged warp: one lane chosen by
// elect.sync executes the instruction.  Keeping the issuing warp converged
// (instead of branching to lane 0) measured 7-11 % faster for the WCSR kernel
// at N <= 128, where the MMA warp's per-item cost bounds the rate.
__device__ __forceinline__ void umma_f16_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The weight-stationary form (M = 32, 64 or 128; N = 64, 128 or 256).  On
// GB300 an M = 64 x N = 256 x K = 16 bf16 MMA takes ~93 cycles in this form
// against 128 in the plain one.  Its M = 64 accumulator holds rows 0..63 in
// TMEM lanes 0..63 for columns 0..N/2-1 and in lanes 64..127 for columns
// N/2..N-1, each in N/2 TMEM columns.
__device__ __forceinline__ void umma_ws_f16_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                  uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.ws.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}
// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk copy global -> shared; completion is reported to `bar` as
// transaction bytes.  x is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Contiguous bulk copy global -> shared (size a multiple of 16 bytes, both
// addresses 16-byte aligned); completion is reported to `bar` as transaction
// bytes.  Runs on the TMA engine, outside the issuing thread's cp.async
// tracking.
__device__ __forceinline__ void tma_bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bring `bytes` of global memory (16-byte aligned, a multiple of 16 bytes)
// into L2 ahead of a later copy, without writing shared memory.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2-D tiled bulk copy shared -> global (a TMA store).  Elements of the box
// outside the tensor are not written.  x is the innermost coordinate and must
// be non-negative with x * element size a multiple of 16 bytes.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of the issuing thread's committed bulk-store groups
// are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until the issuing thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- cp.async
// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros and
// reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

// Arrive on `bar` (without incrementing its pending count) once every
// cp.async this thread issued before has completed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Wait until all of this thread's cp.async copies are complete (the copies
// here are tracked by mbarriers, not commit groups, so wait_all is the form
// that covers them).
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Make this thread's completed generic-proxy shared-memory writes visible to
// the async proxy (tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- cluster launch control
// Asks the hardware to cancel the launch of one CTA of this grid that has not
// started yet; the 16-byte answer is written to `resp` (16-byte aligned
// shared memory) and completes 16 transaction bytes on `bar`, whose phase the
// caller has armed with mbar_arrive_expect_tx(bar, 16).
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
  asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];"
               ::"r"(resp), "r"(bar)
               : "memory");
}

// Reads an answer of clc_try_cancel once its barrier phase has completed:
// true and the cancelled CTA's blockIdx.x, or false when no CTA was left.
__device__ __forceinline__ bool clc_query(uint32_t resp, uint32_t &cta_x) {
  uint32_t ok, x;
  asm volatile(
      "{\n\t.reg .b128 h;\n\t.reg .pred p;\n\t"
      "ld.shared.b128 h, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, h;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, h;\n\t}"
      : "=r"(ok), "=r"(x)
      : "r"(resp)
      : "memory");
  cta_x = x;
  return ok != 0;
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (fp16/bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all tcgen05 operations issued so far by this
// thread have completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp gets lane
// (its sub-partition base + t), columns [col, col+16).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma with 128-byte swizzling.
//   K-major operand (rows of 64 contiguous 16-bit K elements, 128 B apart):
//     lbo unused (16), sbo = 1024 (stride between groups of 8 rows).
//   MN-major operand (64 contiguous M/N elements per K row, 128 B apart):
//     lbo = byte stride between 64-element M/N column groups, sbo = 1024
//     (stride between groups of 8 K rows).
// Tiles must start on a 1024-byte boundary (base offset field 0).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// The descriptor of the same layout `bytes` further on in shared memory
// (bytes a multiple of 16): the start-address field (address / 16, bits
// 0..13) grows by bytes / 16.  Shared-memory addresses stay below 256 KB, so
// the field cannot carry into the next one.
__device__ __forceinline__ uint64_t smem_desc_add(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// Instruction descriptor for tcgen05.mma kind::f16 with fp32 accumulation.
//   ab_bf16: inputs are bf16 (else fp16); a_mn_major / b_mn_major: operand
//   major-ness (0 = K-major); m, n: MMA shape.
__host__ __device__ constexpr uint32_t idesc_f16(bool ab_bf16, bool a_mn_major, bool b_mn_major,
                                                 uint32_t m, uint32_t n) {
  return (1u << 4)                                  // D format: f32
         | ((ab_bf16 ? 1u : 0u) << 7)               // A format
         | ((ab_bf16 ? 1u : 0u) << 10)              // B format
         | ((a_mn_major ? 1u : 0u) << 15)           // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | ((n >> 3) << 17)                         // N / 8
         | ((m >> 4) << 24);                        // M / 16
}

}  // namespace spmm
