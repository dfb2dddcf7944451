// pfa_ptx.cuh -- inline-PTX building blocks for sm_103a: mbarriers, TMA tensor
// loads, and the tcgen05 tensor-core / tensor-memory instructions.
//
// Conventions used throughout the library's kernels:
//  * Shared-memory addresses are 32-bit shared-window addresses (smem_u32).
//  * Tensor-memory (TMEM) addresses are lane << 16 | column, as returned by
//    tcgen05.alloc; a warp may only touch the 32 lanes 32*(warp % 4) .. +31.
//  * Every mbarrier wait is bounded in time: after `limit_ns` it records an
//    error bit, raises the CTA-wide abort flag and returns false.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace pfa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Error bits recorded in the device error word.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrLengths = 2u;  // device-side {T, start_pos} failed its checks

// Graph entry: checks the run-time {T, start_pos} against the capacities the
// grid and the tensor maps were built for.
__device__ __forceinline__ bool lengths_ok(int64_t T, int64_t sp, int64_t max_T, int64_t cap,
                                           int64_t ring_rows, int window) {
  if (T < 0 || T > max_T || sp < 0 || sp + T > ((int64_t)1 << 31) - 4096) return false;
  if (ring_rows == 0) return sp + T <= cap;
  const int64_t span = (int64_t)window + T - 1 < sp + T ? (int64_t)window + T - 1 : sp + T;
  return cap >= span;
}


// Bounded wait for the completion of the phase with parity `parity`.
// Returns true on completion.  Returns false (without completing) when the
// CTA's abort flag is raised, or when `limit_ns` elapses, in which case it
// raises the abort flag and records kErrTimeout in *err.  With
// `ignore_abort` the wait only gives up on the time limit (used to drain
// copies that are known to be in flight before a CTA exits).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* err, uint64_t limit_ns,
                                          bool ignore_abort = false) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 15u) == 0) {
      if (!ignore_abort && *abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

// mbar_wait executed by every lane of a converged warp; the result is the
// same in all lanes (false if any lane gave up).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, unsigned* err,
                                               uint64_t limit_ns, bool ignore_abort = false) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err, limit_ns, ignore_abort));
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 3-D tiled bulk tensor load into this CTA's shared memory; completion is
// signalled on `bar` as transaction bytes.  c0 (innermost) must keep the
// copy 16-byte aligned.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile
// (tcgen05 descriptor format: start >> 4, leading and stride byte offsets
// >> 4, version 1 at bits 46-47, swizzle mode 2 = 128B at bits 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16 with bf16 A/B, fp32 D.
// b_mn_major selects an MN-major (N-contiguous) B operand.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn_major) {
  return (1u << 4)                       // D format: f32
       | (1u << 7)                       // A format: bf16
       | (1u << 10)                      // B format: bf16
       | ((b_mn_major ? 1u : 0u) << 16)  // B major-ness
       | ((uint32_t)(N >> 3) << 17)      // N / 8
       | ((uint32_t)(M >> 4) << 24);     // M / 16
}

// ---- issue from a converged warp: every lane computes the (warp-uniform)
// operands, one elected lane issues.  Keeping the issuing warp converged lets
// the descriptors live in uniform registers; issuing from a lone lane of a
// diverged warp makes every instruction pay for moving its operands.

// Eight K=16 steps of D (+)= A * B with both operands in shared memory.
// Step kk uses descriptors a0 + aoff(kk), b0 + boff(kk), where the offsets are
// in 16-byte units (the descriptor's start-address field):
//   kk = 0..3: + 2 kk,  kk = 4..7: + half + 2 (kk - 4)   (half = 64-column span)
// The first step accumulates iff `accumulate`; the rest always accumulate.
template <uint32_t kHalf16>
__device__ __forceinline__ void mma8_ss_kmajor(uint32_t d_tmem, uint64_t a0, uint64_t b0,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, acc;\n\t.reg .b64 a, b;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 acc, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, acc;\n\t"
      "add.s64 a, %1, 2;  add.s64 b, %2, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, 4;  add.s64 b, %2, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, 6;  add.s64 b, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, %5; add.s64 b, %2, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, %6; add.s64 b, %2, %6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, %7; add.s64 b, %2, %7;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, %8; add.s64 b, %2, %8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t}"
      :: "r"(d_tmem), "l"(a0), "l"(b0), "r"(idesc), "r"(accumulate),
         "n"(kHalf16), "n"(kHalf16 + 2), "n"(kHalf16 + 4), "n"(kHalf16 + 6)
      : "memory");
}

// Eight K=16 steps of D (+)= A * B with A in tensor memory (columns a_tmem +
// 8 kk, packed bf16 pairs) and B in shared memory (descriptor b0 + kk * bstep16,
// offsets in 16-byte units).
template <uint32_t kBStep16>
__device__ __forceinline__ void mma8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, acc;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 acc, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, acc;\n\t"
      "add.s32 a, %1, 8;  add.s64 b, %2, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 16; add.s64 b, %2, %6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 24; add.s64 b, %2, %7;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 32; add.s64 b, %2, %8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 40; add.s64 b, %2, %9;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 48; add.s64 b, %2, %10;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 56; add.s64 b, %2, %11;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b0), "r"(idesc), "r"(accumulate),
         "n"(kBStep16), "n"(2 * kBStep16), "n"(3 * kBStep16), "n"(4 * kBStep16),
         "n"(5 * kBStep16), "n"(6 * kBStep16), "n"(7 * kBStep16)
      : "memory");
}

// Four K=16 steps of D (+)= A * B, both operands K-major in shared memory
// within one 128-byte swizzle span (steps advance both descriptors by 32 B).
__device__ __forceinline__ void mma4_ss_kmajor(uint32_t d_tmem, uint64_t a0, uint64_t b0,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, acc;\n\t.reg .b64 a, b;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 acc, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, acc;\n\t"
      "add.s64 a, %1, 2;  add.s64 b, %2, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, 4;  add.s64 b, %2, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, 6;  add.s64 b, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, e;\n\t}"
      :: "r"(d_tmem), "l"(a0), "l"(b0), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four K=16 steps of D (+)= A * B with A in tensor memory (columns a_tmem +
// 8 kk) and B in shared memory (descriptor b0 + kk * bstep16, 16-byte units).
template <uint32_t kBStep16>
__device__ __forceinline__ void mma4_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, acc;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 acc, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, acc;\n\t"
      "add.s32 a, %1, 8;  add.s64 b, %2, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 16; add.s64 b, %2, %6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 24; add.s64 b, %2, %7;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, e;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b0), "r"(idesc), "r"(accumulate),
         "n"(kBStep16), "n"(2 * kBStep16), "n"(3 * kBStep16)
      : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (tensor core, TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// tcgen05.commit from one elected lane of a converged warp.
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
      :: "r"(bar) : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane -> r[0..31].
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]) : "r"(taddr));
}
// Wait for this thread's outstanding tcgen05.ld; the registers are tied to
// the wait so no use of them can be scheduled above it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- math
// 2^x on the special-function unit (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// Two floats -> packed bf16 pair (round-to-nearest-even); `lo` in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace pfa
