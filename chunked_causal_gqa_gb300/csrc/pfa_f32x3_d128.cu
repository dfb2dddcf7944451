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
// CTA = one kv head x one 128-row query tile (all `group` query heads of the
// kv head for 128/group consecutive tokens; row r -> token r/group, head
// r%group); CTAs in kv-head-major order, latest tokens first within a head.
// Key tiles of 128.
//
// Warp roles (9 warps):
//   warps 0-3  rows of the tile (TMEM lanes 0-127, one row per thread): split
//              Q into hi/lo operand tiles in shared memory once, then the
//              online softmax of every key tile, then the epilogue
//   warps 4-7  converters: read fp32 K and V tiles from global memory (ring
//              and strided caches included), split them into hi/lo bf16 and
//              write the 128-byte-swizzled operand layout a TMA load of a bf16
//              tile would produce, into a 5-slot ring (one slot = one 128x128
//              bf16 tile; a K or V tile takes two slots, hi and lo)
//   warp  8    TMEM allocator and MMA issuer (converged warp, elected lane)
//
// Tensor memory (512 columns): [0,128) S_0 and [128,256) S_1 (double-buffered
// scores; after the softmax P_hi, packed bf16 pairs, fills the first 64
// columns of its buffer), [256,384) O, [384,448) and [448,512) P_lo of the two
// buffers.
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
#include "pfa_ptx.cuh"

#include <cmath>

namespace pfa {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                   // query rows per CTA
constexpr int kBN = 128;                   // keys per tile
constexpr int kThreads = 288;
constexpr int kHalfBytes = 128 * 128;      // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kTileBytes = 2 * kHalfBytes; // 128 rows x 128 bf16
constexpr int kSlots = 5;                  // operand ring depth (bf16 tiles)
constexpr int kSmemQHi = 0;
constexpr int kSmemQLo = kTileBytes;
constexpr int kSmemRing = 2 * kTileBytes;
constexpr int kSmemBars = kSmemRing + kSlots * kTileBytes;  // 229376
constexpr int kSmemAlloc = kSmemBars + 256 + 1024;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// barriers
constexpr int kBarQ = 0;                        // Q hi/lo written (4 row-warp arrivals)
constexpr int kBarFull = 1;                     // kSlots: operand tile written (4 converter arrivals)
constexpr int kBarEmpty = kBarFull + kSlots;    // kSlots: operand tile consumed (commit)
constexpr int kBarS = kBarEmpty + kSlots;       // 2: S(i) complete (commit)
constexpr int kBarP = kBarS + 2;                // 2: P(i) in TMEM (4 row-warp arrivals)
constexpr int kBarO = kBarP + 2;                // O += P(i) V(i) complete (commit), one phase per tile
constexpr int kBarDrain = kBarO + 1;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kOffTmemSlot = kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
static_assert(kOffAbort + 4 <= 256, "barrier area");

constexpr uint32_t kColO = 256, kColPLo = 384;
constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false);  // K-major Q and K
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kD, true);    // V is N(=d)-contiguous

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
// row r in a 128-byte-swizzled K-major bf16 tile of 128 rows x 128 elements:
// 64-element spans 16 KB apart, row r at r * 128, 16-byte chunk c at c ^ (r % 8).
__device__ __forceinline__ uint32_t swz_off(int r, int q) {
  const int span = q >> 4, c = (q & 15) >> 1, half = q & 1;
  return (uint32_t)(span * kHalfBytes + r * 128 + ((c ^ (r & 7)) << 4) + half * 8);
}

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

  // Chunk length and position: kernel parameters, or (graph entry) read from
  // device memory at run time, with the grid sized for the largest T.
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
    if ((int)blockIdx.x >= tiles_per_head * p.Hkv) return;  // nothing set up yet
  }

  // work unit: (kv head, query tile), kv head major, latest tokens first
  // within a head: the CTAs in flight cover few kv heads, so the fp32 K/V
  // they stream (16 MB per head at 16k keys) stays in L2 between them
  const int kh = (int)blockIdx.x / tiles_per_head;
  const int tile = tiles_per_head - 1 - (int)blockIdx.x % tiles_per_head;
  const int64_t t0 = (int64_t)tile * p.tok_per_tile;
  const int64_t t_end = min(t0 + p.tok_per_tile, T);
  const int64_t pos_first = start_pos + t0;
  const int64_t pos_last = start_pos + t_end - 1;
  const int64_t kmin = p.window > 0 ? max((int64_t)0, pos_first - p.window + 1) : 0;
  const int64_t kt_first = kmin / kBN;
  const int n = (int)(pos_last / kBN - kt_first + 1);
  const int64_t L = start_pos + T;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool per_warp = (i == kBarQ || i == kBarP || i == kBarP + 1 ||
                             (i >= kBarFull && i < kBarFull + kSlots));
      mbar_init(bar(i), per_warp ? 4u : 1u);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Ring order (converters and MMA warp), items u = 0 .. 2n-1: K(0); then for
  // i = 1 .. n-1: K(i), V(i-1); then V(n-1).  Each item is two consecutive
  // slot loads: hi, lo.

  if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = mbar_wait_warp(bar(kBarQ), 0, abort_flag, p.err, lim);
    bool issued = false;
    tc_fence_after();
    const uint64_t qhi = sdesc_sw128(sbase + kSmemQHi, 16, 1024);
    const uint64_t qlo = sdesc_sw128(sbase + kSmemQLo, 16, 1024);
    const uint32_t tO = tmem + kColO;
    uint32_t li = 0;  // slot loads consumed
    auto item_ready = [&](uint32_t* s_hi, uint32_t* s_lo) -> bool {
      *s_hi = li % kSlots;
      *s_lo = (li + 1) % kSlots;
      if (!mbar_wait_warp(bar(kBarFull + *s_hi), (li / kSlots) & 1u, abort_flag, p.err, lim))
        return false;
      if (!mbar_wait_warp(bar(kBarFull + *s_lo), ((li + 1) / kSlots) & 1u, abort_flag, p.err,
                          lim))
        return false;
      tc_fence_after();
      li += 2;
      return true;
    };
    auto pv = [&](int j) -> bool {  // O (+)= P(j) V(j): hi*hi + hi*lo + lo*hi
      uint32_t sh, sl;
      if (!item_ready(&sh, &sl)) return false;
      if (!mbar_wait_warp(bar(kBarP + (j & 1)), (uint32_t)(j >> 1) & 1u, abort_flag, p.err, lim))
        return false;
      tc_fence_after();
      const uint32_t tP = tmem + (uint32_t)((j & 1) * kBN);
      const uint64_t vh = sdesc_sw128(sbase + kSmemRing + sh * kTileBytes, kHalfBytes, 1024);
      const uint64_t vl = sdesc_sw128(sbase + kSmemRing + sl * kTileBytes, kHalfBytes, 1024);
      mma8_ts<2048 / 16>(tO, tP, vh, kIdescPV, j > 0 ? 1u : 0u);
      mma8_ts<2048 / 16>(tO, tP, vl, kIdescPV, 1u);
      mma8_ts<2048 / 16>(tO, tmem + kColPLo + (uint32_t)((j & 1) * 64), vh, kIdescPV, 1u);
      tc_commit_elect(bar(kBarEmpty + sh));
      tc_commit_elect(bar(kBarEmpty + sl));
      tc_commit_elect(bar(kBarO));
      return true;
    };
    for (int i = 0; i < n && ok; ++i) {
      // S(i) = Q_hi K_hi + Q_hi K_lo + Q_lo K_hi
      uint32_t sh, sl;
      if (!(ok = item_ready(&sh, &sl))) break;
      const uint32_t tS = tmem + (uint32_t)((i & 1) * kBN);
      const uint64_t kh_d = sdesc_sw128(sbase + kSmemRing + sh * kTileBytes, 16, 1024);
      const uint64_t kl_d = sdesc_sw128(sbase + kSmemRing + sl * kTileBytes, 16, 1024);
      mma8_ss_kmajor<kHalfBytes / 16>(tS, qhi, kh_d, kIdescQK, 0u);
      mma8_ss_kmajor<kHalfBytes / 16>(tS, qhi, kl_d, kIdescQK, 1u);
      mma8_ss_kmajor<kHalfBytes / 16>(tS, qlo, kh_d, kIdescQK, 1u);
      issued = true;
      tc_commit_elect(bar(kBarS + (i & 1)));
      tc_commit_elect(bar(kBarEmpty + sh));
      tc_commit_elect(bar(kBarEmpty + sl));
      if (i > 0 && !(ok = pv(i - 1))) break;
    }
    if (ok) ok = pv(n - 1);
    if (issued) {
      // everything issued must complete before TMEM is freed
      tc_commit_elect(bar(kBarDrain));
      mbar_wait_warp(bar(kBarDrain), 0, abort_flag, p.err, lim, true);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ converters
    // Warp cw converts rows (keys) 32 cw .. 32 cw + 31 of every tile; lane l
    // holds elements 4 l .. 4 l + 3 of a row, so each load is one 512-byte row.
    const int cw = warp - 4;
    const float* kbase = p.k + (int64_t)kh * p.kv_head_stride;
    const float* vbase = p.v + (int64_t)kh * p.kv_head_stride;
    auto row_of = [&](int64_t j) -> int64_t { return p.ring_rows > 0 ? j % p.ring_rows : j; };
    bool ok = true;
    uint32_t li = 0;  // slot loads written
    // Item u of the ring order -> (V?, key tile).
    auto item_of = [&](int u, int* tile) -> bool {
      if (u == 0) { *tile = 0; return false; }
      if (u == 2 * n - 1) { *tile = n - 1; return true; }
      *tile = (u + 1) >> 1;
      if (u & 1) return false;       // u = 2i - 1: K(i)
      *tile = (u >> 1) - 1;          // u = 2i: V(i - 1)
      return true;
    };
    // This warp's 32 rows of item u, as one range of the cache when they are
    // consecutive and written (else nothing: the loads find them in memory).
    auto rows_of = [&](int u, const float** ptr) -> bool {
      int tile;
      const bool is_v = item_of(u, &tile);
      const int64_t key0 = (kt_first + tile) * kBN + cw * 32;
      const int64_t row0 = row_of(key0);
      *ptr = (is_v ? vbase : kbase) + row0 * kD;
      return key0 + 32 <= L && (p.ring_rows == 0 || row0 + 32 <= p.ring_rows);
    };
    auto item = [&](int u) -> bool {
      int tile;
      const float* base = item_of(u, &tile) ? vbase : kbase;
      // Items run ahead of the MMA by about two; ask L2 for the rows of the
      // item after the next now, so that its loads do not wait for DRAM.
      if (u + 2 < 2 * n && lane == 0) {
        const float* pf;
        if (rows_of(u + 2, &pf)) prefetch_l2(pf, 32u * kD * 4u);
      }
      const int64_t key0 = (kt_first + tile) * kBN + cw * 32;
      // Global loads first: their latency overlaps the wait for the slots.
      // Rows past the written keys read as zeros.  The common case (all 32
      // rows written, consecutive in the cache) uses one base pointer.
      float4 x[32];
      const int64_t row0 = row_of(key0);
      if (key0 + 32 <= L && (p.ring_rows == 0 || row0 + 32 <= p.ring_rows)) {
        const float4* src = reinterpret_cast<const float4*>(base + row0 * kD) + lane;
#pragma unroll
        for (int r = 0; r < 32; ++r) x[r] = __ldg(src + r * (kD / 4));
      } else {
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          const int64_t j = key0 + r;
          x[r] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j < L) x[r] = __ldg(reinterpret_cast<const float4*>(base + row_of(j) * kD) + lane);
        }
      }
      const uint32_t s_hi = li % kSlots, s_lo = (li + 1) % kSlots;
      bool good = mbar_wait(bar(kBarEmpty + s_hi), ((li / kSlots) & 1u) ^ 1u, abort_flag, p.err, lim);
      good = good && mbar_wait(bar(kBarEmpty + s_lo), (((li + 1) / kSlots) & 1u) ^ 1u, abort_flag,
                               p.err, lim);
      if (!__all_sync(0xffffffffu, good)) return false;
      uint8_t* hi = smem + kSmemRing + s_hi * kTileBytes;
      uint8_t* lo = smem + kSmemRing + s_lo * kTileBytes;
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        uint2 h, l;
        split4(x[r], &h, &l);
        const uint32_t off = swz_off(cw * 32 + r, lane);
        *reinterpret_cast<uint2*>(hi + off) = h;
        *reinterpret_cast<uint2*>(lo + off) = l;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kBarFull + s_hi));
        mbar_arrive(bar(kBarFull + s_lo));
      }
      li += 2;
      return true;
    };
    if (lane == 0) {
      const float* pf;
      if (rows_of(0, &pf)) prefetch_l2(pf, 32u * kD * 4u);
      if (2 * n > 1 && rows_of(1, &pf)) prefetch_l2(pf, 32u * kD * 4u);
    }
    for (int u = 0; u < 2 * n && ok; ++u) ok = item(u);
  } else {
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
        const uint32_t off = swz_off(row, q4);
        *reinterpret_cast<uint2*>(smem + kSmemQHi + off) = hv;
        *reinterpret_cast<uint2*>(smem + kSmemQLo + off) = lv;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarQ));
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
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          x[j] = __uint_as_float(r0[j]) * c;
          x[32 + j] = __uint_as_float(r1[j]) * c;
          x[64 + j] = __uint_as_float(r2[j]) * c;
          x[96 + j] = __uint_as_float(r3[j]) * c;
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
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t r[32];
        tmem_ld32(tS + 32 * q, r);
        tmem_wait_ld(r);
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float xa = __uint_as_float(r[2 * j]) * c, xb = __uint_as_float(r[2 * j + 1]) * c;
          if (partial) {
            const int ja = 32 * q + 2 * j;
            if (ja > hi_rel || ja <= lo_rel) xa = -INFINITY;
            if (ja + 1 > hi_rel || ja + 1 <= lo_rel) xb = -INFINITY;
          }
          const float pa = ex2(xa - base), pb = ex2(xb - base);
          const uint32_t w = pack_bf16x2(pa, pb);
          ph[j] = w;
          pl[j] = pack_bf16x2(pa - bf16_lo_f32(w), pb - bf16_hi_f32(w));
          ls[(2 * j) & 3] += pa;
          ls[(2 * j + 1) & 3] += pb;
        }
        tmem_st16(tS + 16 * q, ph);
        tmem_st16(tPlo + 16 * q, pl);
      }
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
      if (lane == 0) mbar_arrive(bar(kBarP + (i & 1)));
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

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_f32x3_d128(const Call& c) {
  static DeviceOnce setup;
  const int sr = setup.run(c.device, [] {
    return cudaFuncSetAttribute(f32x3_d128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemAlloc) == cudaSuccess ? kOk : kErrLaunch;
  });
  if (sr != kOk) return sr;
  const int group = c.H / c.Hkv;
  const int tok_per_tile = kBM / group;
  const int64_t tiles = (c.T + tok_per_tile - 1) / tok_per_tile;
  const int64_t L = c.start_pos + c.T;
  if (tiles * c.Hkv > 0x7fffffff || L + kBN > 0x7fffffff) return kErrShape;
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
  f32x3_d128_kernel<<<dim3((unsigned)(tiles * c.Hkv)), kThreads, kSmemAlloc, c.stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace pfa
