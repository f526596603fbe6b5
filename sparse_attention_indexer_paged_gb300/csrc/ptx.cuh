// Inline-PTX building blocks for sm_103a: mbarriers, TMA (cp.async.bulk),
// tcgen05 MMA / TMEM, and bounded waits that never hang the GPU.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "common.cuh"

namespace dsa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test (acquire on success): has the phase with this parity
// completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The test the bounded waits repeat: mbarrier.try_wait without a time hint
// may suspend the thread for a system-dependent time before returning false
// (measured 3 % faster in the logits kernel than an explicit 0.1 ms hint,
// and no slower than pure polling).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  return mbar_try_wait(bar, parity);
}

// Wait until the phase of `bar` with the given parity has completed.  Returns
// false (without waiting further) once the CTA's abort flag is set, or after
// kWaitTimeoutNs, in which case it records DSA_ERR_TIMEOUT and sets the flag
// so that every other role of the CTA stops too.
__device__ __forceinline__ bool wait_or_abort_for(uint32_t bar, uint32_t parity,
                                                  volatile int32_t* abort_flag, int32_t* status,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      report(status, kErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int32_t* abort_flag, int32_t* status) {
  return wait_or_abort_for(bar, parity, abort_flag, status, kWaitTimeoutNs);
}

// Bounded wait that ignores the abort flag: used while draining copies that
// are already in flight before the CTA exits.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_sleep(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainTimeoutNs) return false;
  }
  return true;
}

// Programmatic dependent launch: wait until the kernel this one was launched
// after has completed and its memory is visible (a no-op without that launch
// attribute); let the kernel launched after this one start its set-up.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One lane of the (fully converged) warp is chosen; true on that lane only.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// 16-byte asynchronous global -> shared copy (completes in the background;
// the issuing thread waits for it with cp_async_wait).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most `n` of this thread's committed copy groups are pending.
template <int n>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

// ---------------------------------------------------------------- TMA / bulk copies

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 2-D tiled TMA load into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int32_t x,
                                            int32_t y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 3-D tiled TMA load into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int32_t x,
                                            int32_t y, int32_t z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// Plain bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05 / TMEM

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

// Shared-memory matrix descriptor of a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart
// (stride byte offset), descriptor version 1, layout code 2 (SWIZZLE_128B).
// The tile must start on a 1024-byte boundary; a K offset inside the
// 128-byte row is added to the start address.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor: D fp32, A and B of the given format code, both
// K-major, shape M x N.
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format,
//   15/16 A/B major (0 = K), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc(uint32_t a_fmt, uint32_t b_fmt, uint32_t M,
                                             uint32_t N) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t kFmtE4M3 = 0;  // kind::f8f6f4
constexpr uint32_t kFmtF16 = 0;   // kind::f16

__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc_v, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc_v), "r"(accumulate)
      : "memory");
}

// As mma_f8f6f4 with each descriptor given as its two 32-bit halves (the
// pair is assembled inside the asm, so no 64-bit arithmetic is needed), and
// the accumulate flag fixed at compile time.
template <bool kAccumulate>
__device__ __forceinline__ void mma_f8f6f4_w(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                             uint32_t b_lo, uint32_t b_hi, uint32_t idesc_v) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc_v), "n"(kAccumulate ? 1 : 0)
      : "memory");
}

template <bool kAccumulate>
__device__ __forceinline__ void mma_f16_w(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                          uint32_t b_lo, uint32_t b_hi, uint32_t idesc_v) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc_v), "n"(kAccumulate ? 1 : 0)
      : "memory");
}

// A 128-deep contraction as one block of MMAs into d_tmem (the first step
// overwrites, the rest accumulate); only threads with `issue` set issue it
// (one elected lane of the MMA warp).  K-major operands with the 128-byte
// swizzle: inside a 128-byte row a 32-byte K step is +2 in the descriptor's
// address field.
//   e4m3 (kind::f8f6f4): four K = 32 steps inside one 128-byte row.
__device__ __forceinline__ void mma_fp8_k128(uint32_t issue, uint32_t d_tmem, uint32_t a_lo,
                                             uint32_t b_lo, uint32_t hi, uint32_t idesc_v) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b64 da, db;\n\t.reg .b32 al, bl;\n\t"
      "setp.ne.b32 p, %0, 0;\n\t"
      "setp.ne.b32 f, %4, %4;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "mov.b64 da, {%2, %4};\n\tmov.b64 db, {%3, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%1], da, db, %5, f;\n\t"
      "add.u32 al, %2, 2;\n\tadd.u32 bl, %3, 2;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%1], da, db, %5, t;\n\t"
      "add.u32 al, %2, 4;\n\tadd.u32 bl, %3, 4;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%1], da, db, %5, t;\n\t"
      "add.u32 al, %2, 6;\n\tadd.u32 bl, %3, 6;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%1], da, db, %5, t;\n\t}" ::"r"(issue),
      "r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc_v)
      : "memory");
}

//   f16 (kind::f16): eight K = 16 steps; elements 0-63 and 64-127 sit in two
//   separate swizzled blocks (the A block of a 128-token tile is 16 KB, the B
//   block of the Q rows is kFp4QHalfBytes), four steps inside each.
constexpr uint32_t kFp4AHalfLo = (128 * 128) >> 4;
// b_half_lo: the distance of the B operand's second k-half (the pass's q rows) >> 4
__device__ __forceinline__ void mma_f16_k128(uint32_t issue, uint32_t d_tmem, uint32_t a_lo,
                                             uint32_t b_lo, uint32_t hi, uint32_t idesc_v, uint32_t b_half_lo) {
  const uint32_t a2 = a_lo + kFp4AHalfLo, b2 = b_lo + b_half_lo;
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b64 da, db;\n\t.reg .b32 al, bl;\n\t"
      "setp.ne.b32 p, %0, 0;\n\t"
      "setp.ne.b32 f, %4, %4;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "mov.b64 da, {%2, %4};\n\tmov.b64 db, {%3, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, f;\n\t"
      "add.u32 al, %2, 2;\n\tadd.u32 bl, %3, 2;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t"
      "add.u32 al, %2, 4;\n\tadd.u32 bl, %3, 4;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t"
      "add.u32 al, %2, 6;\n\tadd.u32 bl, %3, 6;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t"
      "mov.b64 da, {%6, %4};\n\tmov.b64 db, {%7, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t"
      "add.u32 al, %6, 2;\n\tadd.u32 bl, %7, 2;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t"
      "add.u32 al, %6, 4;\n\tadd.u32 bl, %7, 4;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t"
      "add.u32 al, %6, 6;\n\tadd.u32 bl, %7, 6;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %5, t;\n\t}" ::"r"(issue),
      "r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc_v), "r"(a2), "r"(b2)
      : "memory");
}

// ---------------------------------------------------------------- block-scaled e2m1 (kind::mxf4)
// Packed e2m1 operands (two elements a byte, K-major, 64-byte rows) stored
// with the 64-byte swizzle: 8-row groups of 512 bytes (stride byte offset),
// layout code 4.  High word of the shared-memory descriptor:
constexpr uint32_t kSdescHiSw64 = (512 >> 4) | (1u << 14) | (4u << 29);

// Instruction descriptor of kind::mxf4 (scale_vec::2X, ue8m0 scales): A and
// B e2m1 (format code 1 at bits 7-9 and 10-12), D always f32, bit 23 = ue8m0
// scale format, N >> 3 at bits 17-22, M >> 4 at bits 24-28; the scale-factor
// ids (which byte of each 32-bit scale word the instruction starts at) sit at
// bits 29-30 (A) and 4-5 (B).
__host__ __device__ constexpr uint32_t idesc_mxf4(uint32_t M, uint32_t N) {
  return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

// Scale factors in TMEM for kind::mxf4: the scales of operand row x (a key
// token of A, a column of B) are the 32-bit word at lane x mod 32 -- the
// same in every lane quarter -- and column base + x / 32; byte i of the word
// scales K block i (32 elements) of the row.  One 128-row block is 32 lanes x
// 4 columns, filled from 512 bytes of shared memory by one copy that
// replicates to the four lane quarters: TMEM lane l, column c <- the 32-bit
// word 4 l + c of the source.  So the source holds row x's word at
// 4 (x mod 32) + x / 32.
//
// Shared-memory descriptor of that source (no swizzle: 8-row x 16-byte core
// matrices of 128 contiguous bytes, both strides 128 bytes):
__device__ __forceinline__ uint32_t sdesc_lo_plain(uint32_t saddr) {
  return ((saddr >> 4) & 0x3FFFu) | ((128u >> 4) << 16);
}
constexpr uint32_t kSdescHiPlain = (128 >> 4) | (1u << 14);

// tcgen05.cp of one 512-byte scale block to TMEM (32 lanes x 128 bits, to
// all four lane quarters), by the threads with `issue` set.  It runs in issue
// order with the same thread's MMAs, and a later commit covers it.
__device__ __forceinline__ void tmem_cp_scales(uint32_t issue, uint32_t taddr, uint32_t s_lo, uint32_t s_hi) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 d;\n\t"
      "setp.ne.b32 p, %0, 0;\n\t"
      "mov.b64 d, {%2, %3};\n\t"
      "@p tcgen05.cp.cta_group::1.32x128b.warpx4 [%1], d;\n\t}" ::"r"(issue),
      "r"(taddr), "r"(s_lo), "r"(s_hi)
      : "memory");
}

// A 128-deep block-scaled e2m1 contraction into d_tmem: two K = 64 steps,
// each 32 bytes into the operands' 64-byte rows (+2 in the descriptor's
// address field); the first takes scale bytes 0-1 (K blocks 0 and 1) and
// overwrites, the second takes bytes 2-3 (scale-factor id 2 for A and B)
// and accumulates.  sfa / sfb: TMEM addresses of the two operands' scales.
__device__ __forceinline__ void mma_mxf4_k128(uint32_t issue, uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                              uint32_t hi, uint32_t idesc_v, uint32_t sfa, uint32_t sfb) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b64 da, db;\n\t.reg .b32 al, bl, id2;\n\t"
      "setp.ne.b32 p, %0, 0;\n\t"
      "setp.ne.b32 f, %4, %4;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "mov.b64 da, {%2, %4};\n\tmov.b64 db, {%3, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%1], da, db, %5, [%6], [%7], f;\n\t"
      "add.u32 al, %2, 2;\n\tadd.u32 bl, %3, 2;\n\t"
      "or.b32 id2, %5, 0x40000020;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%1], da, db, id2, [%6], [%7], t;\n\t}" ::"r"(issue),
      "r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc_v), "r"(sfa), "r"(sfb)
      : "memory");
}

// tcgen05.commit by the threads with `issue` set.
__device__ __forceinline__ void mma_commit_if(uint32_t issue, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}" ::"r"(issue),
      "r"(bar)
      : "memory");
}

// Orders this thread's shared-memory writes before later async-proxy reads
// (tcgen05.mma operands) that are ordered after it by an mbarrier.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four bytes, each holding two e2m1 values (element 2i in the low nibble),
// to four f16x2 words (lower half = the low nibble's value).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

// Two e4m3 codes (the first in the low byte) to an f16x2 word (low half = first).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(two_bytes)));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// High and low 32-bit words of sdesc_k_sw128(saddr).
constexpr uint32_t kSdescHi = (1024 >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr) { return ((saddr >> 4) & 0x3FFFu) | (1u << 16); }

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc_v, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc_v), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 64 columns of 32-bit TMEM words: thread i of the warp receives
// lane (taddr.lane + i), columns taddr.col .. taddr.col + 63.
__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM words (as tmem_ld_x64, half the columns).
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 columns of 32-bit TMEM words.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld_x16(taddr, r); }
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld_x32(taddr, r); }
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[64]) { tmem_ld_x64(taddr, r); }

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace dsa
