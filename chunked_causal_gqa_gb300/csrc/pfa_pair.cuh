// pfa_pair.cuh -- inline-PTX building blocks for kernels whose two CTAs of a
// cluster issue their tensor-core products together (tcgen05 cta_group::2):
// cluster addressing and arrivals, bounded cluster-scope waits, TMA loads that
// complete on the peer's barrier, the paired tensor-memory allocation, the
// M = 256 products and their multicast commits.
//
// In a kernel that uses these, every tcgen05 instruction that takes a CTA
// group uses cta_group::2: the allocation is made by one warp of each CTA of
// the pair, the products are issued by rank 0 and read both CTAs' shared and
// tensor memory (each CTA supplies its own rows of A and half of B, and its
// tensor memory receives its own rows of D), and a commit arrives on the
// mbarrier at the given offset in each CTA of the mask.  Measured on GB300:
// an mbarrier arrival with release at cluster scope costs the arriving
// thread ~1.2k cycles; the arrivals here use the default (CTA-scope)
// release, like the tensor-core pipeline's own signals, and the waits
// acquire at cluster scope.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "pfa_ptx.cuh"

namespace pfa {


__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of both CTAs: orders earlier shared-memory work (barrier
// initialisation, remote arrivals) before the peer's later accesses.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// Arrival on an mbarrier given by its cluster address (this CTA's or the
// peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" :: "r"(cluster_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// mbar_wait for a barrier the peer CTA arrives on (acquire at cluster
// scope), executed by every lane of a converged warp; bounded in time like
// every other wait.
__device__ __forceinline__ bool mbar_wait_cl_warp(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, unsigned* err,
                                                  uint64_t limit_ns) {
  bool ok = mbar_try_wait_cl(bar, parity);
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
      if (mbar_try_wait_cl(bar, parity)) {
        ok = true;
        break;
      }
      if ((spin & 15u) == 0) {
        if (*abort_flag) break;
        if (globaltimer_ns() - t0 > limit_ns) {
          *abort_flag = 1;
          atomicOr(err, kErrTimeout);
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// 3-D tiled bulk tensor load into this CTA's shared memory whose completion
// is signalled, as transaction bytes, on an mbarrier of either CTA of the
// pair (given by its cluster address).  c0 must keep the copy 16-byte aligned.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cluster_bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}

// Eight K=16 steps of D (+)= A * B for the pair, both operands K-major in
// 128-byte-swizzled tiles: steps 0-3 in the spans at a0 / b0, steps 4-7 in
// the spans kAHalf16 / kBHalf16 further (16-byte units).  From one converged
// warp; one elected lane issues.
template <uint32_t kAHalf16, uint32_t kBHalf16>
__device__ __forceinline__ void mma8_ss_pair(uint32_t d_tmem, uint64_t a0, uint64_t b0,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, acc;\n\t.reg .b64 a, b;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 acc, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, acc;\n\t"
      "add.s64 a, %1, 2;  add.s64 b, %2, 2;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, 4;  add.s64 b, %2, 4;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, 6;  add.s64 b, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, %5;  add.s64 b, %2, %9;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, %6;  add.s64 b, %2, %10;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, %7;  add.s64 b, %2, %11;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, e;\n\t"
      "add.s64 a, %1, %8;  add.s64 b, %2, %12;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, e;\n\t}"
      :: "r"(d_tmem), "l"(a0), "l"(b0), "r"(idesc), "r"(accumulate),
         "n"(kAHalf16), "n"(kAHalf16 + 2), "n"(kAHalf16 + 4), "n"(kAHalf16 + 6),
         "n"(kBHalf16), "n"(kBHalf16 + 2), "n"(kBHalf16 + 4), "n"(kBHalf16 + 6)
      : "memory");
}

// Four K=16 steps of D (+)= A * B for the pair, A in tensor memory (columns
// a_tmem + 8 kk, packed bf16 pairs) and B in shared memory (descriptor b0 +
// kk * kBStep16, 16-byte units).
template <uint32_t kBStep16>
__device__ __forceinline__ void mma4_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, acc;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 acc, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, acc;\n\t"
      "add.s32 a, %1, 8;  add.s64 b, %2, %5;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 16; add.s64 b, %2, %6;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 24; add.s64 b, %2, %7;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b0), "r"(idesc), "r"(accumulate),
         "n"(kBStep16), "n"(2 * kBStep16), "n"(3 * kBStep16)
      : "memory");
}

// Eight K=16 steps of D (+)= A * B for the pair, A in tensor memory (columns
// a_tmem + 8 kk, packed bf16 pairs) and B in shared memory (descriptor b0 +
// kk * kBStep16, 16-byte units).
template <uint32_t kBStep16>
__device__ __forceinline__ void mma8_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, acc;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 acc, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, acc;\n\t"
      "add.s32 a, %1, 8;  add.s64 b, %2, %5;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 16; add.s64 b, %2, %6;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 24; add.s64 b, %2, %7;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 32; add.s64 b, %2, %8;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 40; add.s64 b, %2, %9;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 48; add.s64 b, %2, %10;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t"
      "add.s32 a, %1, 56; add.s64 b, %2, %11;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, e;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b0), "r"(idesc), "r"(accumulate),
         "n"(kBStep16), "n"(2 * kBStep16), "n"(3 * kBStep16), "n"(4 * kBStep16),
         "n"(5 * kBStep16), "n"(6 * kBStep16), "n"(7 * kBStep16)
      : "memory");
}

// Commit of the issuing thread's earlier products, arriving on the mbarrier
// at offset `bar` in both CTAs of the pair.  From one converged warp.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}"
      :: "r"(bar), "h"((uint16_t)3) : "memory");
}

// 32 bytes (eight 32-bit words) to a 32-byte aligned global address.
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                  "r"(w[6]), "r"(w[7])
               : "memory");
}

}  // namespace pfa
