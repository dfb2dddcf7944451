// pfa_f32x3_d128.cu -- fp32 prefill attention, head_dim 128, on the sm_103a
// bf16 tensor cores with a three-product split of every operand.
//
// Operation (gnosis "Prefill attention -> GPU: handoff", section "GPU design",
// steps 1-3, fused; accuracy bar max |gpu - cpu| <= 1e-4 of its section
// "Implementation status"): per query row, scores against the visible keys of
// its kv head, scale, causal (+ window) mask, softmax, weighted sum of V.
//
// Precision.  One bf16 value keeps 8 significant bits, far too few for the
// 1e-4 bar.  Every fp32 operand x is split into hi = bf16(x) and
// lo = bf16(x - hi) (both rounded to nearest even; x - hi is exact in fp32), so
// |x - hi - lo| <= 2^-18 |x|.  Each contraction is formed as
//     hi*hi + hi*lo + lo*hi
// on tcgen05.mma kind::f16 (a product of two bf16 values is exact in fp32;
// fp32 accumulation in tensor memory).  The dropped lo*lo term and the
// rounding of lo leave ~2^-17 relative per product: a CPU emulation of the
// scheme on the tiny fp32 layer stays at 1.5e-5 of the oracle, and the
// three-product tf32 form it replaces needed the tf32 rate, half the bf16
// rate, on operands twice as large.
//
// Pairs of CTAs.  The two CTAs of a cluster (ranks 0 and 1, on two SMs) take
// query tiles 2p and 2p + 1 of one kv head (each: all `group` query heads for
// 128/group consecutive tokens; row r -> token r/group, head r%group), and
// rank 0 issues products of M = 256 rows for both (tcgen05.mma.cta_group::2):
// each CTA supplies its own query rows and half of the B operand -- keys
// 64 r .. 64 r + 63 of each K tile, columns 64 r .. 64 r + 63 of each V tile
// -- so each SM converts half of every fp32 K and V tile.  (With one CTA per
// tile, each SM converted whole tiles, and the conversion, not the tensor
// core, set the pace.)  The pair walks the union of its two tiles' key
// ranges; each CTA masks the keys its own rows do not see.  Clusters in
// kv-head-major order, latest tokens first within a head.  Key tiles of 128.
//
// Warp roles (9 warps per CTA):
//   warps 0-3  rows of the tile (TMEM lanes 0-127, one row per thread): split
//              Q into hi/lo operand tiles in shared memory once, then the
//              online softmax of every key tile, then the epilogue
//   warps 4-7  converters: read this CTA's half of the fp32 K and V tiles
//              from global memory (ring and strided caches included), split
//              them into hi/lo bf16 and write the 128-byte-swizzled operand
//              layout a TMA load of a bf16 tile would produce, into a ring of
//              5 items (an item: hi and lo of one K or V half, 32 KB)
//   warp  8    TMEM allocation (both ranks); on rank 0 the MMA issuer
//              (converged warp, elected lane)
// Rank 0's barriers for operands, Q and P count the arrivals of both CTAs'
// warps; rank 0's commits arrive on the barrier at the same offset in both.
//
// Tensor memory (each CTA, 512 columns): [0,128) S_0 and [128,256) S_1
// (double-buffered scores; after the softmax P_hi, packed bf16 pairs, fills
// the first 64 columns of its buffer), [256,384) O, [384,448) and [448,512)
// P_lo of the two buffers.
//
// MMA issue order: S(0), S(1), O += P(0) V(0), S(2), O += P(1) V(1), ...
// so that while the softmax of tile i runs, the tensor core executes
// O += P(i-1) V(i-1) and S(i+1).  The softmax of tile i waits for
// O += P(i-1) V(i-1) (barrier kBarO, one phase per tile) before it may rescale O.
//
// Online softmax in the log2 domain with the lazy rescale of the other
// kernels (the exponent base rises only when a row maximum exceeds it by more
// than 2^8); masks come from indices; every wait is bounded.
#include "pfa_internal.h"
#include "pfa_pair.cuh"
#include "pfa_ptx.cuh"

#include <cmath>

namespace pfa {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                   // query rows per CTA
constexpr int kBN = 128;                   // keys per tile
constexpr int kThreads = 288;
constexpr int kHalfBytes = 128 * 128;      // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kTileBytes = 2 * kHalfBytes; // 128 rows x 128 bf16 (the Q operand tiles)
constexpr int kPartBytes = 16384;          // one CTA's half of a K or V operand tile (hi or lo)
constexpr int kKSpan = 8192;               // K half: 64 keys x 64 columns per 128-byte span
constexpr int kItems = 5;                  // operand ring depth (items: hi + lo of a K or V half)
constexpr int kItemBytes = 2 * kPartBytes;
constexpr int kSmemQHi = 0;
constexpr int kSmemQLo = kTileBytes;
constexpr int kSmemRing = 2 * kTileBytes;
constexpr int kSmemBars = kSmemRing + kItems * kItemBytes;  // 229376
constexpr int kSmemAlloc = kSmemBars + 256 + 1024;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// barriers (rank 0's count both CTAs' arrivals; rank 1's kBarQ, kBarFull and
// kBarP are unused)
constexpr int kBarQ = 0;                        // Q hi/lo written (8 row-warp arrivals)
constexpr int kBarFull = 1;                     // kItems: operand item written (8 converter arrivals)
constexpr int kBarEmpty = kBarFull + kItems;    // kItems: operand item consumed (commit)
constexpr int kBarS = kBarEmpty + kItems;       // 2: S(i) complete (commit)
constexpr int kBarP = kBarS + 2;                // 2: P(i) in TMEM (8 row-warp arrivals)
constexpr int kBarO = kBarP + 2;                // O += P(i) V(i) complete (commit), one phase per tile
constexpr int kBarDrain = kBarO + 1;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kOffTmemSlot = kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
static_assert(kOffAbort + 4 <= 256, "barrier area");

constexpr uint32_t kColO = 256, kColPLo = 384;
constexpr uint32_t kIdescQK = idesc_bf16_f32(2 * kBM, kBN, false);  // K-major Q and K
constexpr uint32_t kIdescPV = idesc_bf16_f32(2 * kBM, kD, true);    // V is N(=d)-contiguous

struct Params {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  int64_t qkv_dim;           // elements from one token's q / out row to the next
  int64_t kv_head_stride;    // elements from one kv head's cache block to the next
  int64_t ring_rows;         // > 0: key j is in cache row j % ring_rows; 0: in row j
  int64_t T, start_pos;      // graph entry: T = the largest T, start_pos unused
  const int64_t* lens;       // graph entry: device {T, start_pos}; else null
  int64_t kv_capacity;       // rows per kv head in the cache
  int H, Hkv, group, tok_per_tile, window, tiles_per_head;
  float scale_log2;
  unsigned* err;
  uint64_t wait_limit_ns;
  int flags;
};

// fp32 of the bf16 in the low / high half of a packed pair.
__device__ __forceinline__ float bf16_lo_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Pairs of fp32 values in one 64-bit register, and the packed pair
// arithmetic of sm_100+ (each lane rounded as its scalar counterpart).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Four consecutive fp32 values -> (hi, lo) as two packed bf16 pairs each.
__device__ __forceinline__ void split4(const float4 x, uint2* hi, uint2* lo) {
  const uint32_t h01 = pack_bf16x2(x.x, x.y), h23 = pack_bf16x2(x.z, x.w);
  hi->x = h01;
  hi->y = h23;
  lo->x = pack_bf16x2(x.x - bf16_lo_f32(h01), x.y - bf16_hi_f32(h01));
  lo->y = pack_bf16x2(x.z - bf16_lo_f32(h23), x.w - bf16_hi_f32(h23));
}

// 16 consecutive 32-bit TMEM columns of this thread's lane <- r[0..15].
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                  "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
                  "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}

// Asks L2 to fetch `bytes` (a multiple of 16) from global memory at `ptr`
// (16-byte aligned); no data reaches the SM and nothing has to be waited for.
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
               :: "l"(reinterpret_cast<uint64_t>(ptr)), "r"(bytes) : "memory");
}

// Byte offset of the 8-byte piece holding elements 4q .. 4q+3 (q = 0..31) of
// row r in a 128-byte-swizzled K-major bf16 tile of `rows` rows x 128
// elements: 64-element spans rows * 128 bytes apart, row r at r * 128, 16-byte
// chunk c at c ^ (r % 8).
template <int kRows>
__device__ __forceinline__ uint32_t swz_off(int r, int q) {
  const int span = q >> 4, c = (q & 15) >> 1, half = q & 1;
  return (uint32_t)(span * (kRows * 128) + r * 128 + ((c ^ (r & 7)) << 4) + half * 8);
}

// kPosScale (scale > 0): the row maximum is taken over the unscaled scores and
// scaled once, which leaves the order of the scores unchanged.
template <bool kPosScale>
__global__ void __launch_bounds__(kThreads, 1) f32x3_d128_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kSmemBars;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemBars + kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemBars + kOffAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int rank = (int)cluster_ctarank();  // = blockIdx.x & 1 (clusters of two)

  // Chunk length and position: kernel parameters, or (graph entry) read from
  // device memory at run time, with the grid sized for the largest T.  Both
  // CTAs of a cluster take every decision below from the same values.
  int64_t T = p.T, start_pos = p.start_pos;
  int tiles_per_head = p.tiles_per_head;
  if (p.lens) {
    T = p.lens[0];
    start_pos = p.lens[1];
    if (!lengths_ok(T, start_pos, p.T, p.kv_capacity, p.ring_rows, p.window)) {
      if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, kErrLengths);
      return;
    }
    tiles_per_head = (int)((T + p.tok_per_tile - 1) / p.tok_per_tile);
  }
  const int pairs_per_head = (tiles_per_head + 1) / 2;
  const int cl = (int)(blockIdx.x >> 1);
  if (p.lens && cl >= pairs_per_head * p.Hkv) return;  // nothing set up yet

  // Unit of cluster cl: (kv head, pair of query tiles), kv head major, latest
  // tokens first within a head: the clusters in flight cover few kv heads, so
  // the fp32 K/V they stream (16 MB per head at 16k keys) stays in L2
  // between them.  This CTA's tile is 2 pair + rank (past T for the second
  // tile of an odd last pair: its rows hold no token).
  const int kh = cl / pairs_per_head;
  const int pair = pairs_per_head - 1 - cl % pairs_per_head;
  const int64_t t0 = (int64_t)(2 * pair + rank) * p.tok_per_tile;
  const int64_t t0a = (int64_t)(2 * pair) * p.tok_per_tile;
  const int64_t t_end = min(t0a + 2 * (int64_t)p.tok_per_tile, T);  // end of the pair's tokens
  const int64_t kmin = p.window > 0 ? max((int64_t)0, start_pos + t0a - p.window + 1) : 0;
  const int64_t kt_first = kmin / kBN;
  const int n = (int)((start_pos + t_end - 1) / kBN - kt_first + 1);
  const int64_t L = start_pos + T;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool per_warp = (i == kBarQ || i == kBarP || i == kBarP + 1 ||
                             (i >= kBarFull && i < kBarFull + kItems));
      mbar_init(bar(i), per_warp ? 8u : 1u);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t bar0 = cluster_addr(bars, 0);  // rank 0's barrier area
  auto bar_r0 = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

  // Ring order (converters and MMA warp), items u = 0 .. 2n-1: K(0); then for
  // i = 1 .. n-1: K(i), V(i-1); then V(n-1).  Item u occupies ring entry
  // u % kItems: hi at its start, lo 16 KB further.

  if (warp == 8 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    bool ok = mbar_wait_cl_warp(bar(kBarQ), 0, abort_flag, p.err, lim);
    bool issued = false;
    tc_fence_after();
    const uint64_t qhi = sdesc_sw128(sbase + kSmemQHi, 16, 1024);
    const uint64_t qlo = sdesc_sw128(sbase + kSmemQLo, 16, 1024);
    const uint32_t tO = tmem + kColO;
    uint32_t ui = 0;  // items consumed
    auto item_ready = [&](uint32_t* e) -> bool {
      *e = ui % kItems;
      if (!mbar_wait_cl_warp(bar(kBarFull + (int)*e), (ui / kItems) & 1u, abort_flag, p.err, lim))
        return false;
      tc_fence_after();
      ++ui;
      return true;
    };
    auto pv = [&](int j) -> bool {  // O (+)= P(j) V(j): hi*hi + hi*lo + lo*hi
      uint32_t e;
      if (!item_ready(&e)) return false;
      if (!mbar_wait_cl_warp(bar(kBarP + (j & 1)), (uint32_t)(j >> 1) & 1u, abort_flag, p.err, lim))
        return false;
      tc_fence_after();
      const uint32_t tP = tmem + (uint32_t)((j & 1) * kBN);
      const uint32_t ib = sbase + kSmemRing + e * kItemBytes;
      // this CTA's 64 columns of V: one 128-byte span, 16 keys per step (2048 B)
      const uint64_t vh = sdesc_sw128(ib, kKSpan, 1024);
      const uint64_t vl = sdesc_sw128(ib + kPartBytes, kKSpan, 1024);
      mma8_ts_pair<2048 / 16>(tO, tP, vh, kIdescPV, j > 0 ? 1u : 0u);
      mma8_ts_pair<2048 / 16>(tO, tP, vl, kIdescPV, 1u);
      mma8_ts_pair<2048 / 16>(tO, tmem + kColPLo + (uint32_t)((j & 1) * 64), vh, kIdescPV, 1u);
      tc_commit_pair(bar(kBarEmpty + (int)e));
      tc_commit_pair(bar(kBarO));
      return true;
    };
    for (int i = 0; i < n && ok; ++i) {
      // S(i) = Q_hi K_hi + Q_hi K_lo + Q_lo K_hi
      uint32_t e;
      if (!(ok = item_ready(&e))) break;
      const uint32_t tS = tmem + (uint32_t)((i & 1) * kBN);
      const uint32_t ib = sbase + kSmemRing + e * kItemBytes;
      const uint64_t kh_d = sdesc_sw128(ib, 16, 1024);
      const uint64_t kl_d = sdesc_sw128(ib + kPartBytes, 16, 1024);
      mma8_ss_pair<kHalfBytes / 16, kKSpan / 16>(tS, qhi, kh_d, kIdescQK, 0u);
      mma8_ss_pair<kHalfBytes / 16, kKSpan / 16>(tS, qhi, kl_d, kIdescQK, 1u);
      mma8_ss_pair<kHalfBytes / 16, kKSpan / 16>(tS, qlo, kh_d, kIdescQK, 1u);
      issued = true;
      tc_commit_pair(bar(kBarS + (i & 1)));
      tc_commit_pair(bar(kBarEmpty + (int)e));
      if (i > 0 && !(ok = pv(i - 1))) break;
    }
    if (ok) ok = pv(n - 1);
    if (issued) {
      // everything issued must complete before either CTA frees its TMEM
      tc_commit_pair(bar(kBarDrain));
      mbar_wait_warp(bar(kBarDrain), 0, abort_flag, p.err, lim, true);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ converters
    // K item: this CTA's keys 64 rank .. +63 of the tile; warp cw converts 16
    // of them, lane l holding elements 4 l .. 4 l + 3 of a row (one 512-byte
    // row per load).  V item: columns 64 rank .. +63 of all 128 keys; warp cw
    // converts keys 32 cw .. 32 cw + 31, two rows per load (lanes 0-15 and
    // 16-31, lane l holding columns 64 rank + 4 (l % 16) .. + 3).
    const int cw = warp - 4;
    const float* kbase = p.k + (int64_t)kh * p.kv_head_stride;
    const float* vbase = p.v + (int64_t)kh * p.kv_head_stride;
    auto row_of = [&](int64_t j) -> int64_t { return p.ring_rows > 0 ? j % p.ring_rows : j; };
    bool ok = true;
    uint32_t ui = 0;  // items written
    // Item u of the ring order -> (V?, key tile).
    auto item_of = [&](int u, int* tile) -> bool {
      if (u == 0) { *tile = 0; return false; }
      if (u == 2 * n - 1) { *tile = n - 1; return true; }
      *tile = (u + 1) >> 1;
      if (u & 1) return false;       // u = 2i - 1: K(i)
      *tile = (u >> 1) - 1;          // u = 2i: V(i - 1)
      return true;
    };
    // First key and row count of this warp's part of item u.
    auto part_of = [&](int u, bool* is_v) -> int64_t {
      int tile;
      *is_v = item_of(u, &tile);
      const int64_t key0 = (kt_first + tile) * kBN;
      return *is_v ? key0 + 32 * cw : key0 + 64 * rank + 16 * cw;
    };
    // Asks L2 for the rows of this warp's part of item u (whole rows; only
    // when they are written and consecutive in the cache).
    auto prefetch_part = [&](int u) {
      bool is_v;
      const int64_t k0 = part_of(u, &is_v);
      const int rows = is_v ? 32 : 16;
      const int64_t r0 = row_of(k0);
      if (k0 + rows <= L && (p.ring_rows == 0 || r0 + rows <= p.ring_rows))
        prefetch_l2((is_v ? vbase : kbase) + r0 * kD, (uint32_t)rows * kD * 4u);
    };
    auto item = [&](int u) -> bool {
      // Items run ahead of the MMA by about two; ask L2 for the rows of the
      // item after the next now, so that its loads do not wait for DRAM.
      if (u + 2 < 2 * n && lane == 0) prefetch_part(u + 2);
      bool is_v;
      const int64_t k0 = part_of(u, &is_v);
      // Global loads first: their latency overlaps the wait for the entry.
      // Rows past the written keys read as zeros.
      float4 x[16];
      if (!is_v) {
        const float* src = kbase + lane * 4;
        const int64_t r0 = row_of(k0);
        if (k0 + 16 <= L && (p.ring_rows == 0 || r0 + 16 <= p.ring_rows)) {
#pragma unroll
          for (int r = 0; r < 16; ++r) x[r] = __ldg(reinterpret_cast<const float4*>(src + (r0 + r) * kD));
        } else {
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            x[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k0 + r < L) x[r] = __ldg(reinterpret_cast<const float4*>(src + row_of(k0 + r) * kD));
          }
        }
      } else {
        const float* src = vbase + 64 * rank + 4 * (lane & 15);
        const int64_t r0 = row_of(k0);
        const int sub = lane >> 4;  // row 2 r + sub
        if (k0 + 32 <= L && (p.ring_rows == 0 || r0 + 32 <= p.ring_rows)) {
#pragma unroll
          for (int r = 0; r < 16; ++r)
            x[r] = __ldg(reinterpret_cast<const float4*>(src + (r0 + 2 * r + sub) * kD));
        } else {
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const int64_t j = k0 + 2 * r + sub;
            x[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < L) x[r] = __ldg(reinterpret_cast<const float4*>(src + row_of(j) * kD));
          }
        }
      }
      const uint32_t e = ui % kItems;
      const bool good = mbar_wait(bar(kBarEmpty + (int)e), ((ui / kItems) & 1u) ^ 1u, abort_flag,
                                  p.err, lim);
      if (!__all_sync(0xffffffffu, good)) return false;
      uint8_t* hi = smem + kSmemRing + e * kItemBytes;
      uint8_t* lo = hi + kPartBytes;
      if (!is_v) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          uint2 h, l;
          split4(x[r], &h, &l);
          const uint32_t off = swz_off<64>(16 * cw + r, lane);
          *reinterpret_cast<uint2*>(hi + off) = h;
          *reinterpret_cast<uint2*>(lo + off) = l;
        }
      } else {
        // MN-major: key j at j * 128, 16-byte chunk c (columns 8c .. 8c+7 of
        // this CTA's 64) at c ^ (j % 8)
        const int c = (lane & 15) >> 1, half = lane & 1;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const int j = 32 * cw + 2 * r + (lane >> 4);
          uint2 h, l;
          split4(x[r], &h, &l);
          const uint32_t off = (uint32_t)(j * 128 + ((c ^ (j & 7)) << 4) + half * 8);
          *reinterpret_cast<uint2*>(hi + off) = h;
          *reinterpret_cast<uint2*>(lo + off) = l;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(bar_r0(kBarFull + (int)e));
      ++ui;
      return true;
    };
    if (lane == 0) {
      prefetch_part(0);
      if (2 * n > 1) prefetch_part(1);
    }
    for (int u = 0; u < 2 * n && ok; ++u) ok = item(u);
  } else if (warp < 4) {
    // ------------------------------------------------------------ rows
    const int row = threadIdx.x;  // = TMEM lane
    const int tok = row / p.group;
    const int hrow = row % p.group;
    const bool row_exists = tok < p.tok_per_tile;
    const int64_t t = t0 + tok;
    const bool row_valid = row_exists && t < T;
    const int h = kh * p.group + hrow;
    const int64_t pos = start_pos + t;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float c = p.scale_log2;

    // Q row -> hi / lo operand tiles (rows that hold no token stay zero)
    {
      const float4* qrow = reinterpret_cast<const float4*>(p.q + t * p.qkv_dim + (int64_t)h * kD);
#pragma unroll 4
      for (int q4 = 0; q4 < 32; ++q4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row_valid) x = __ldg(qrow + q4);
        uint2 hv, lv;
        split4(x, &hv, &lv);
        const uint32_t off = swz_off<128>(row, q4);
        *reinterpret_cast<uint2*>(smem + kSmemQHi + off) = hv;
        *reinterpret_cast<uint2*>(smem + kSmemQLo + off) = lv;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(bar_r0(kBarQ));
    }

    bool ok = true;
    if (p.flags & kFlagForceTimeout) {
      // Test hook: wait on a barrier nothing signals, so the limit expires.
      ok = mbar_wait(bar(kBarDrain), 0, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    const uint32_t tO = tmem + lane_off + kColO;
    float m_run = -INFINITY, l = 0.f;
    for (int i = 0; i < n && ok; ++i) {
      ok = mbar_wait(bar(kBarS + (i & 1)), (uint32_t)(i >> 1) & 1u, abort_flag, p.err, lim);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + (uint32_t)((i & 1) * kBN);
      const uint32_t tPlo = tmem + lane_off + kColPLo + (uint32_t)((i & 1) * 64);
      // key j of the tile is visible iff j <= hi_rel and j > lo_rel
      const int64_t key0 = (kt_first + i) * kBN;
      const int hi_rel = (int)(pos - key0);
      const int lo_rel = p.window > 0 ? (int)(pos - p.window - key0) : -1;
      const bool partial = hi_rel < kBN - 1 || lo_rel >= 0;
      // Two passes over the scores in tensor memory: the row maximum first,
      // then P 32 keys at a time (fewer live registers than one pass).
      float mx;
      {
        float x[128];
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(tS, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_wait_ld(r0);
        tmem_wait_ld(r1);
        tmem_wait_ld(r2);
        tmem_wait_ld(r3);
        const float cs = kPosScale ? 1.f : c;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          x[j] = __uint_as_float(r0[j]) * cs;
          x[32 + j] = __uint_as_float(r1[j]) * cs;
          x[64 + j] = __uint_as_float(r2[j]) * cs;
          x[96 + j] = __uint_as_float(r3[j]) * cs;
        }
        if (partial) {
#pragma unroll
          for (int j = 0; j < 128; ++j)
            if (j > hi_rel || j <= lo_rel) x[j] = -INFINITY;
        }
        float m[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) m[q] = max3f(x[q], x[8 + q], x[16 + q]);
#pragma unroll
        for (int j = 24; j < 120; j += 16) {
#pragma unroll
          for (int q = 0; q < 8; ++q) m[q] = max3f(m[q], x[j + q], x[j + 8 + q]);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) m[q] = fmaxf(m[q], x[120 + q]);
        mx = max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
        if (kPosScale) mx *= c;
      }
      // Raise the exponent base only when the new maximum exceeds it by > 2^8.
      float alpha = 1.f;
      bool rescale = false;
      if (mx > m_run + kRescaleThreshold) {
        alpha = ex2(m_run - mx);  // 0 while nothing was accumulated
        rescale = (i > 0) && (m_run != -INFINITY);
        m_run = mx;
      }
      const float base = (m_run == -INFINITY) ? 0.f : m_run;
      // P = 2^(s - base) split into hi / lo bf16 pairs, 32 keys at a time:
      // P_hi over the first 64 columns of this tile's scores (chunk q lands
      // in columns of chunk q / 2, already read), P_lo in its own columns;
      // l gains the row sum of the fp32 values (4 independent partial sums)
      // Arithmetic on packed pairs of keys (2j, 2j+1): s c - base, the
      // residual p - hi, and the row sums (lanes of ls2[0]: even pairs' keys
      // 2j and 2j+1, of ls2[1]: odd pairs')
      const uint64_t c2 = f2_pack(c, c), nb2 = f2_pack(-base, -base);
      uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t r[32];
        tmem_ld32(tS + 32 * q, r);
        tmem_wait_ld(r);
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float xa, xb;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), c2, nb2),
                    xa, xb);
          if (partial) {
            const int ja = 32 * q + 2 * j;
            if (ja > hi_rel || ja <= lo_rel) xa = -INFINITY;
            if (ja + 1 > hi_rel || ja + 1 <= lo_rel) xb = -INFINITY;
          }
          const float pa = ex2(xa), pb = ex2(xb);
          const uint32_t w = pack_bf16x2(pa, pb);
          ph[j] = w;
          const uint64_t pab = f2_pack(pa, pb);
          float da, db;
          f2_unpack(f2_sub(pab, f2_pack(bf16_lo_f32(w), bf16_hi_f32(w))), da, db);
          pl[j] = pack_bf16x2(da, db);
          ls2[j & 1] = f2_add(ls2[j & 1], pab);
        }
        tmem_st16(tS + 16 * q, ph);
        tmem_st16(tPlo + 16 * q, pl);
      }
      float ls[4];
      f2_unpack(ls2[0], ls[0], ls[1]);
      f2_unpack(ls2[1], ls[2], ls[3]);
      l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      if (i > 0) {
        // O is stable once O += P(i-1) V(i-1) has completed.
        ok = mbar_wait(bar(kBarO), (uint32_t)(i - 1) & 1u, abort_flag, p.err, lim);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st32(tO + c0, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(bar_r0(kBarP + (i & 1)));
    }
    if (ok) {
      ok = mbar_wait(bar(kBarO), (uint32_t)(n - 1) & 1u, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* orow = p.out + t * p.qkv_dim + (int64_t)h * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c0, o);
        tmem_wait_ld(o);
        if (row_valid) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(orow + c0 + 4 * j) =
                make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                            __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
        }
      }
    }
  }

  // Neither CTA leaves, nor frees tensor memory, while the pair's products
  // may still touch it: rank 0 drains them before this point.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

int launch_f32x3_d128(const Call& c) {
  static DeviceOnce setup;
  const int sr = setup.run(c.device, [] {
    if (cudaFuncSetAttribute(f32x3_d128_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemAlloc) != cudaSuccess)
      return kErrLaunch;
    return cudaFuncSetAttribute(f32x3_d128_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemAlloc) == cudaSuccess ? kOk : kErrLaunch;
  });
  if (sr != kOk) return sr;
  const int group = c.H / c.Hkv;
  const int tok_per_tile = kBM / group;
  const int64_t tiles = (c.T + tok_per_tile - 1) / tok_per_tile;
  const int64_t pairs = (tiles + 1) / 2;
  const int64_t L = c.start_pos + c.T;
  if (2 * pairs * c.Hkv > 0x7fffffff || L + 2 * kBN > 0x7fffffff) return kErrShape;
  Params p;
  p.q = static_cast<const float*>(c.q);
  p.k = static_cast<const float*>(c.k);
  p.v = static_cast<const float*>(c.v);
  p.out = static_cast<float*>(c.out);
  p.qkv_dim = c.qkv_dim;
  p.kv_head_stride = c.max_seq_len * (int64_t)kD;
  p.ring_rows = ring_rows(c);
  p.T = c.T;
  p.start_pos = c.start_pos;
  p.lens = c.lens;
  p.kv_capacity = c.max_seq_len;
  p.H = c.H;
  p.Hkv = c.Hkv;
  p.group = group;
  p.tok_per_tile = tok_per_tile;
  p.window = c.window;
  p.tiles_per_head = (int)tiles;
  p.scale_log2 = (float)((double)c.scale * 1.4426950408889634);
  p.err = c.err;
  p.wait_limit_ns = c.wait_limit_ns;
  p.flags = c.flags;
  // Clusters of two consecutive CTAs: the two query tiles of a pair.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs * c.Hkv));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = p.scale_log2 > 0.f ? cudaLaunchKernelEx(&cfg, f32x3_d128_kernel<true>, p)
                                             : cudaLaunchKernelEx(&cfg, f32x3_d128_kernel<false>, p);
  if (e != cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return kErrLaunch;
  return kOk;
}

}  // namespace pfa
