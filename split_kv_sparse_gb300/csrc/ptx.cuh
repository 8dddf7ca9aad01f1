// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// (tiled and tile::gather4) loads, tcgen05 TMEM allocation / MMA / commit /
// load / store, and the shared-memory matrix descriptors the MMAs read.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace skv {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity (never suspends the thread,
// unlike try_wait); for a thread that polls several barriers in turn.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Everything a bounded wait needs: a time limit, the kernel's status word and
// a per-CTA abort flag in shared memory that lets one stuck role stop the others.
struct WaitCtx {
  uint64_t limit_ns;
  uint32_t* status;         // global: [0] = MLA_STATUS_* bits, [1] = first site that timed out
  volatile int* abort_flag; // shared
};

// The waiting part of wait_bounded, out of line: the common case (the phase
// has already completed) costs no call.
static __device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, const WaitCtx& ctx,
                                               uint32_t site) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    // polled with test_wait: measured a little faster than a suspending try_wait
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*ctx.abort_flag) return false;
      if (globaltimer_ns() - t0 > ctx.limit_ns) {
        *ctx.abort_flag = 1;
        atomicOr(&ctx.status[0], 1u);
        atomicCAS(&ctx.status[1], 0u, site);
        return false;
      }
    }
  }
}

// Waits for the phase with the given parity of `bar`. Gives up after
// ctx.limit_ns (or when another role of this CTA has aborted), records the
// timeout in the status word and returns false. Never traps. The first test
// never suspends the thread (a suspending try_wait could sit out a wait of any
// length inside the hardware's own window, where no limit is checked).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& ctx, uint32_t site) {
  if (mbar_test_wait(bar, parity)) return true;
  return wait_bounded_slow(bar, parity, ctx, site);
}

// ------------------------------------------------- flags in global memory --

// Load with acquire semantics at GPU scope: reads after it see what the writer
// published before its release.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Store with release semantics at GPU scope.
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------------------------------- fences --

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the OR of `v` over the participating threads
// (a reduction in the barrier itself, with no shared-memory traffic).
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n"
      "  .reg .pred p, q;\n"
      "  setp.ne.u32 q, %1, 0;\n"
      "  bar.red.or.pred p, %2, %3, q;\n"
      "  selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ------------------------------------------- programmatic dependent launch --

// Lets the next kernel in the stream (launched with programmatic serialisation)
// start its launch now; it still waits in grid_dependency_wait() for this grid.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Blocks until the preceding grid has completed and its memory is visible
// (returns at once when the kernel was not launched as a dependent).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Requests one 2-D box of a tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const void* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Bulk shared -> global copy (async proxy), bytes a multiple of 16, both addresses
// 16-byte aligned; tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait_all() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ----------------------------------------------------------------- cp.async --

// 16-byte global -> shared copy through L2 (L1 bypassed); src_bytes = 0 writes
// 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// The same with a constant byte offset folded into the source address.
template <int kOff>
__device__ __forceinline__ void cp_async_16_off(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1+%3], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes), "n"(kOff)
               : "memory");
}
// ... with constant offsets on both addresses.
template <int kDstOff, int kSrcOff>
__device__ __forceinline__ void cp_async_16_off2(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0+%3], [%1+%4], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes),
               "n"(kDstOff), "n"(kSrcOff)
               : "memory");
}
// Bulk global -> shared copy (TMA engine), completion counted on `bar` in bytes;
// both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
               "l"(gsrc), "r"(bytes), "r"(bar)
               : "memory");
}
// Orders this thread's earlier memory accesses (any state space, generic proxy)
// before its later async-proxy operations.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Starts bringing `bytes` (a multiple of 16) at a 16-byte aligned global address
// into L2; no completion to wait for.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Requests the 128-byte line holding `p` into L2 (no completion to wait for).
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Arrives on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05 --

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
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, one instruction of kind::f16 (bf16 or f16 inputs, fp32 D).
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with each operand descriptor given as its two 32-bit words. The low
// word holds the start-address field, so stepping an operand through a tile is
// one 32-bit add; the high words of every 128-byte-swizzled operand with an
// 8-row atom stride of 1024 bytes are equal, so one register serves both.
__device__ __forceinline__ void mma_f16_w(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t ab_hi,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  .reg .b64 da, db;\n"
      "  setp.ne.b32 p, %5, 0;\n"
      "  mov.b64 da, {%1, %3};\n"
      "  mov.b64 db, {%2, %3};\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(ab_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with a compile-time accumulate flag (folded into the predicate).
template <int kAccumulate>
__device__ __forceinline__ void mma_f16_wc(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t ab_hi,
                                           uint32_t idesc) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  .reg .b64 da, db;\n"
      "  setp.ne.b32 p, %5, 0;\n"
      "  mov.b64 da, {%1, %3};\n"
      "  mov.b64 db, {%2, %3};\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(ab_hi), "r"(idesc), "n"(kAccumulate)
      : "memory");
}

// Same for 8-bit inputs (kind::f8f6f4; e4m3 x e4m3 with fp32 D).
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kind::f8f6f4 with each operand descriptor as its two 32-bit words (see
// mma_f16_w) and a compile-time accumulate flag.
template <int kAccumulate>
__device__ __forceinline__ void mma_f8_wc(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t ab_hi,
                                          uint32_t idesc) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  .reg .b64 da, db;\n"
      "  setp.ne.b32 p, %5, 0;\n"
      "  mov.b64 da, {%1, %3};\n"
      "  mov.b64 db, {%2, %3};\n"
      "  tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %4, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(ab_hi), "r"(idesc), "n"(kAccumulate)
      : "memory");
}

// Arrives once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// The same, issued only when `cond` is non-zero: a predicated instruction, not a
// branch, so a run of MMAs around it stays one straight stream.
__device__ __forceinline__ void mma_commit_if(uint32_t bar, uint32_t cond) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  setp.ne.b32 p, %1, 0;\n"
      "  @p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
      "}\n" ::"r"(bar),
      "r"(cond)
      : "memory");
}

#include "tmem_ldst.inc"

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   K-major operand: rows of 128 B (64 bf16 / 128 fp8 of K) in 8-row atoms of
//     1024 B; sbo = byte stride between 8-row atoms; lbo unused (16).
//   MN-major operand: 128 B of MN per K row, 8 K rows per 1024-B atom;
//     lbo = byte stride between 64-element MN atoms, sbo = stride between 8-row K atoms.
// Bits: [0,14) start >> 4, [16,30) lbo >> 4, [32,46) sbo >> 4, [46,49) = 0b001,
// [61,64) swizzle mode (2 = 128 B).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Descriptor of an operand without swizzling (8-row x 16-byte core matrices):
// lbo = byte stride between core matrices along K, sbo = along M/N.
__device__ __forceinline__ uint64_t sdesc_noswizzle(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor: fp32 accumulator, A/B element format `fmt`
// (kind::f16: 0 = f16, 1 = bf16; kind::f8f6f4: 0 = e4m3), operand majorness,
// M and N. Bits: [4,6) D format (1 = f32), [7,10) A fmt, [10,13) B fmt,
// 15 A MN-major, 16 B MN-major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_make(int M, int N, uint32_t fmt, bool a_mn, bool b_mn) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace skv
