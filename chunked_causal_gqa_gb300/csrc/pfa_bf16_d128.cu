// pfa_bf16_d128.cu -- fused flash-style prefill attention for bf16, head_dim 128,
// on the sm_103a tensor cores (tcgen05 + tensor memory + TMA).
//
// Operation (gnosis "Prefill attention -> GPU: handoff", section "GPU design",
// steps 1-3, fused): per query row, scores against the visible keys of its kv
// head, scale, causal (+ window) mask, softmax, weighted sum of V.
//
// Work unit (one CTA): one kv head and two consecutive 128-row query tiles,
// A and B.  A tile packs all `group` query heads of the kv head for
// 128 / group consecutive tokens (row r -> token r / group, head r % group),
// so every K/V tile that TMA brings into shared memory feeds all heads of the
// GQA group, and both tiles.
//
// Warp roles (10 warps):
//   warps 0-3  softmax for tile A (TMEM lanes 0-127, one row per thread)
//   warps 4-7  softmax for tile B
//   warp  8    TMA producer: Q tiles once, then K/V tiles into a 5-slot ring
//   warp  9    TMEM allocator and single-thread tcgen05.mma issuer
//
// Tensor memory (512 columns x 128 lanes, fp32 cells):
//   [  0,128) S_A = Q_A K^T ; after softmax its first 64 columns hold P_A as
//             packed bf16 pairs, the A operand of P_A V
//   [128,256) S_B / P_B
//   [256,384) O_A accumulator      [384,512) O_B accumulator
//
// MMA issue order per key tile i (single issuing thread, executed in order):
//   S_A(i) = Q_A K_i^T, O_B += P_B(i-1) V_{i-1}, S_B(i) = Q_B K_i^T, O_A += P_A(i) V_i
// While the softmax warps of one tile work, the tensor core runs the other
// tile's products.  Because S_X(i) is issued after O_X += P_X(i-1) V, the
// commit that signals S_X(i) also guarantees that product is complete, so the
// softmax warps may rescale O_X and overwrite P_X without a further barrier.
//
// Online softmax in the log2 domain (scores pre-multiplied by scale*log2 e).
// The running maximum used as the exponent base is only raised when a new
// row maximum exceeds it by more than 2^8, so O is rescaled rarely; the final
// normalisation O / l is exact for any base.  l is summed from the same
// bf16-rounded P that feeds the P V product.
//
// Masks come from indices: key j is visible to a row at position pos iff
// j <= pos and (window <= 0 or j > pos - window).  Key tiles outside every
// row's band are never loaded; tiles fully inside every row's band skip the
// per-element test.
#include "pfa_internal.h"
#include "pfa_ptx.cuh"

#include <cuda_bf16.h>

#include <cmath>

namespace pfa {
namespace {

constexpr int kBM = 128;                        // rows per query tile
constexpr int kBN = 128;                        // keys per K/V tile
constexpr int kHalfBytes = 128 * 128;           // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kTileBytes = 2 * kHalfBytes;      // 128 rows x 128 bf16
constexpr int kSlots = 5;                       // K/V ring depth (tiles)
constexpr int kThreads = 320;
constexpr float kRescaleThreshold = 8.0f;       // log2 units

constexpr int kSmemQ = 0;                                   // Q_A, Q_B
constexpr int kSmemRing = 2 * kTileBytes;
constexpr int kSmemBars = kSmemRing + kSlots * kTileBytes;  // 229376
constexpr int kSmemUsed = kSmemBars + 256;
constexpr int kSmemAlloc = kSmemUsed + 1024;                // + alignment slack

// barrier indices (8 bytes each, from kSmemBars)
constexpr int kBarQ = 0;
constexpr int kBarFull = 1;                  // kSlots
constexpr int kBarEmpty = kBarFull + kSlots; // kSlots
constexpr int kBarS = kBarEmpty + kSlots;    // 2 (A, B)
constexpr int kBarP = kBarS + 2;             // 2
constexpr int kBarO = kBarP + 2;             // 2
constexpr int kBarDrain = kBarO + 2;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kOffTmemSlot = kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
static_assert(kOffAbort + 4 <= 256, "barrier area");

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false);  // K-major Q and K
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, 128, true);   // V is N(=d)-contiguous

struct Params {
  __nv_bfloat16* out;
  int64_t T, start_pos;
  int H, Hkv, group, tok_per_tile, window, units_per_head;
  float scale_log2;
  unsigned* err;
  uint64_t wait_limit_ns;
  int flags;
};

struct Unit {
  int kh;
  int64_t t0A, t0B;
  int64_t kt_first;  // first key tile
  int n;             // number of key tiles
};

__device__ __forceinline__ Unit unit_of(const Params& p, int b) {
  Unit u;
  u.kh = b % p.Hkv;
  const int idx = p.units_per_head - 1 - b / p.Hkv;  // latest tokens (most keys) first
  u.t0A = (int64_t)(2 * idx) * p.tok_per_tile;
  u.t0B = u.t0A + p.tok_per_tile;
  const int64_t t_end = min(u.t0B + p.tok_per_tile, p.T);  // exclusive, > t0A
  const int64_t pos_lo = p.start_pos + u.t0A;
  const int64_t pos_hi = p.start_pos + t_end - 1;
  const int64_t kmin = p.window > 0 ? max((int64_t)0, pos_lo - p.window + 1) : 0;
  u.kt_first = kmin / kBN;
  u.n = (int)(pos_hi / kBN - u.kt_first + 1);
  return u;
}

// 8 MMAs (K = 16 each) of S = Q K^T over d = 0..127.
__device__ __forceinline__ void issue_qk(uint32_t tS, uint32_t q_addr, uint32_t k_addr) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_ss(tS, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
           kIdescQK, kk > 0 ? 1u : 0u);
  }
}
// 8 MMAs (K = 16 keys each) of O (+)= P V, P read from tensor memory.
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint32_t v_addr,
                                         bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    // 16 keys = two 8-row groups (SBO 1024 B); d = 0..127 spans the two
    // 64-column halves of the tile (LBO = one half).
    mma_ts(tO, tP + kk * 8, sdesc_sw128(v_addr + kk * 2048, kHalfBytes, 1024), kIdescPV,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <bool kFoldScale>
__global__ void __launch_bounds__(kThreads, 1)
bf16_d128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kSmemBars;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemBars + kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemBars + kOffAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Unit u = unit_of(p, blockIdx.x);
  const uint64_t lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kBarS + x), 1);
      mbar_init(bar(kBarP + x), 4);  // one arrival per softmax warp
      mbar_init(bar(kBarO + x), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int hq = u.kh * p.group;
      // Each Q box is group x tok_per_tile rows of 128 bytes (zero-filled past T).
      const uint32_t q_bytes = 4u * 128u * (uint32_t)(p.group * p.tok_per_tile);
      mbar_arrive_expect_tx(bar(kBarQ), q_bytes);
      tma_load_3d(sbase + kSmemQ, &tm_q, bar(kBarQ), 0, hq, (int)u.t0A);
      tma_load_3d(sbase + kSmemQ + kHalfBytes, &tm_q, bar(kBarQ), 64, hq, (int)u.t0A);
      tma_load_3d(sbase + kSmemQ + kTileBytes, &tm_q, bar(kBarQ), 0, hq, (int)u.t0B);
      tma_load_3d(sbase + kSmemQ + kTileBytes + kHalfBytes, &tm_q, bar(kBarQ), 64, hq,
                  (int)u.t0B);
      uint32_t li = 0;
      bool ok = true;
      for (int i = 0; i < u.n && ok; ++i) {
        const int key0 = (int)((u.kt_first + i) * kBN);
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t s = li % kSlots, ph = (li / kSlots) & 1u;
          if (!mbar_wait(bar(kBarEmpty + s), ph ^ 1u, abort_flag, p.err, lim)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + kSmemRing + s * kTileBytes;
          const CUtensorMap* map = kv ? &tm_v : &tm_k;
          mbar_arrive_expect_tx(bar(kBarFull + s), kTileBytes);
          tma_load_3d(dst, map, bar(kBarFull + s), 0, key0, u.kh);
          tma_load_3d(dst + kHalfBytes, map, bar(kBarFull + s), 64, key0, u.kh);
          ++li;
        }
      }
      (void)ok;
      // No copy may be in flight when the CTA exits.  On the normal path the
      // MMA thread has already consumed every load, so these return at once.
      mbar_wait(bar(kBarQ), 0, abort_flag, p.err, lim, true);
      const uint32_t first = li > (uint32_t)kSlots ? li - kSlots : 0;
      for (uint32_t j = first; j < li; ++j)
        mbar_wait(bar(kBarFull + j % kSlots), (j / kSlots) & 1u, abort_flag, p.err, lim, true);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tSA = tmem + 0, tSB = tmem + 128, tOA = tmem + 256, tOB = tmem + 384;
      const uint32_t qA = sbase + kSmemQ, qB = sbase + kSmemQ + kTileBytes;
      bool ok = mbar_wait(bar(kBarQ), 0, abort_flag, p.err, lim);
      tc_fence_after();
      uint32_t li = 0;  // ring index of K_i
      bool issued = false;
      for (int i = 0; i < u.n && ok; ++i) {
        const uint32_t ks = li % kSlots;
        if (!(ok = mbar_wait(bar(kBarFull + ks), (li / kSlots) & 1u, abort_flag, p.err, lim)))
          break;
        tc_fence_after();
        const uint32_t k_addr = sbase + kSmemRing + ks * kTileBytes;
        issue_qk(tSA, qA, k_addr);
        issued = true;
        tc_commit(bar(kBarS + 0));
        if (i > 0) {
          if (!(ok = mbar_wait(bar(kBarP + 1), (uint32_t)(i - 1) & 1u, abort_flag, p.err, lim)))
            break;
          tc_fence_after();
          const uint32_t vs = (li - 1) % kSlots;  // V_{i-1}
          issue_pv(tOB, tSB, sbase + kSmemRing + vs * kTileBytes, i - 1 > 0);
          tc_commit(bar(kBarEmpty + vs));
        }
        issue_qk(tSB, qB, k_addr);
        tc_commit(bar(kBarS + 1));
        tc_commit(bar(kBarEmpty + ks));
        const uint32_t vs = (li + 1) % kSlots;  // V_i
        if (!(ok = mbar_wait(bar(kBarFull + vs), ((li + 1) / kSlots) & 1u, abort_flag, p.err, lim)))
          break;
        if (!(ok = mbar_wait(bar(kBarP + 0), (uint32_t)i & 1u, abort_flag, p.err, lim))) break;
        tc_fence_after();
        issue_pv(tOA, tSA, sbase + kSmemRing + vs * kTileBytes, i > 0);
        li += 2;
      }
      if (ok) {
        ok = mbar_wait(bar(kBarP + 1), (uint32_t)(u.n - 1) & 1u, abort_flag, p.err, lim);
        if (ok) {
          tc_fence_after();
          const uint32_t vs = (li - 1) % kSlots;
          issue_pv(tOB, tSB, sbase + kSmemRing + vs * kTileBytes, u.n - 1 > 0);
          tc_commit(bar(kBarEmpty + vs));
          tc_commit(bar(kBarO + 0));
          tc_commit(bar(kBarO + 1));
        }
      }
      if (issued) {
        // Everything issued must complete before TMEM is freed (this matters
        // when another role gave up early and skipped its wait on kBarO).
        tc_commit(bar(kBarDrain));
        mbar_wait(bar(kBarDrain), 0, abort_flag, p.err, lim, true);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int X = warp >> 2;        // 0: tile A, 1: tile B
    const int wq = warp & 3;        // lane quarter
    const int row = wq * 32 + lane;
    const int64_t t0 = X ? u.t0B : u.t0A;
    const int tok = row / p.group;
    const bool row_exists = tok < p.tok_per_tile;
    const int64_t t = t0 + tok;
    const bool row_valid = row_exists && t < p.T;
    const int64_t pos = p.start_pos + t;
    const int h = u.kh * p.group + row % p.group;
    const int64_t pos_first = p.start_pos + t0;
    const int64_t pos_last = pos_first + p.tok_per_tile - 1;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)(X * 128);
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(X * 128);
    const float c = p.scale_log2;

    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    if ((p.flags & kFlagForceTimeout) && X == 0) {
      // Test hook: wait on a barrier nothing signals, so the limit expires.
      ok = mbar_wait(bar(kBarDrain), 0, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    for (int i = 0; i < u.n && ok; ++i) {
      ok = mbar_wait(bar(kBarS + X), (uint32_t)i & 1u, abort_flag, p.err, lim);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();

      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(tS + 0, r0);
      tmem_ld32(tS + 32, r1);
      tmem_ld32(tS + 64, r2);
      tmem_ld32(tS + 96, r3);
      tmem_wait_ld(r0);
      tmem_wait_ld(r1);
      tmem_wait_ld(r2);
      tmem_wait_ld(r3);
      float x[128];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = __uint_as_float(r0[j]);
        x[32 + j] = __uint_as_float(r1[j]);
        x[64 + j] = __uint_as_float(r2[j]);
        x[96 + j] = __uint_as_float(r3[j]);
      }
      if (!kFoldScale) {
#pragma unroll
        for (int j = 0; j < 128; ++j) x[j] *= c;
      }
      const int64_t key0 = (u.kt_first + i) * kBN;
      const bool all_visible = (key0 + kBN - 1 <= pos_first) &&
                               (p.window <= 0 || key0 > pos_last - p.window);
      if (!all_visible) {
        const int64_t hi = pos - key0;                                   // j - key0 <= hi
        const int64_t lo = p.window > 0 ? pos - p.window - key0 : -1;    // j - key0 > lo
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j > hi || j <= lo) x[j] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 128; ++j) mx = fmaxf(mx, x[j]);
      if (kFoldScale) mx *= c;

      // Raise the exponent base only when the new maximum exceeds it by > 2^8.
      float alpha = 1.f;
      bool rescale = false;
      if (mx > m_run + kRescaleThreshold) {
        alpha = ex2(m_run - mx);  // 0 while nothing was accumulated
        rescale = (i > 0) && (m_run != -INFINITY);
        m_run = mx;
      }
      const float base = (m_run == -INFINITY) ? 0.f : m_run;

      uint32_t pk0[32], pk1[32];
      float lsum = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float a, b;
        if (kFoldScale) {
          a = ex2(fmaf(x[2 * j], c, -base));
          b = ex2(fmaf(x[2 * j + 1], c, -base));
        } else {
          a = ex2(x[2 * j] - base);
          b = ex2(x[2 * j + 1] - base);
        }
        pk0[j] = pack_bf16x2(a, b);
        lsum += bf16_lo(pk0[j]) + bf16_hi(pk0[j]);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float a, b;
        if (kFoldScale) {
          a = ex2(fmaf(x[64 + 2 * j], c, -base));
          b = ex2(fmaf(x[64 + 2 * j + 1], c, -base));
        } else {
          a = ex2(x[64 + 2 * j] - base);
          b = ex2(x[64 + 2 * j + 1] - base);
        }
        pk1[j] = pack_bf16x2(a, b);
        lsum += bf16_lo(pk1[j]) + bf16_hi(pk1[j]);
      }
      l = l * alpha + lsum;

      // O_X is stable here: the commit that signalled S_X(i) covers P_X(i-1) V.
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st32(tO + c0, o);
        }
      }
      tmem_st32(tS + 0, pk0);
      tmem_st32(tS + 32, pk1);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarP + X));
    }

    if (ok) {
      ok = mbar_wait(bar(kBarO + X), 0, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.out + ((t * p.H + h) * (int64_t)128);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c0, o);
        tmem_wait_ld(o);
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_bf16_d128(const Call& c) {
  static int attr_done[64] = {0};
  if (c.device < 0 || c.device >= 64) return kErrDevice;
  if (!attr_done[c.device]) {
    if (cudaFuncSetAttribute(bf16_d128_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemAlloc) != cudaSuccess ||
        cudaFuncSetAttribute(bf16_d128_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemAlloc) != cudaSuccess)
      return kErrLaunch;
    attr_done[c.device] = 1;
  }
  const int group = c.H / c.Hkv;
  const int tok_per_tile = kBM / group;  // group <= 128 checked by the caller
  const int64_t tiles = (c.T + tok_per_tile - 1) / tok_per_tile;
  const int64_t units = (tiles + 1) / 2;
  const int64_t L = c.start_pos + c.T;
  if (units * c.Hkv > 0x7fffffff || L + kBN > 0x7fffffff ||
      c.T + 2 * (int64_t)tok_per_tile > 0x7fffffff)
    return kErrShape;

  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {128, (uint64_t)c.H, (uint64_t)c.T};
    const uint64_t strides[2] = {128 * 2, (uint64_t)c.H * 128 * 2};
    const uint32_t box[3] = {64, (uint32_t)group, (uint32_t)tok_per_tile};
    if (encode_tmap_bf16_3d(&tq, c.q, dims, strides, box)) return kErrLaunch;
  }
  {
    const uint64_t dims[3] = {128, (uint64_t)L, (uint64_t)c.Hkv};
    const uint64_t strides[2] = {128 * 2, (uint64_t)L * 128 * 2};
    const uint32_t box[3] = {64, (uint32_t)kBN, 1};
    if (encode_tmap_bf16_3d(&tk, c.k, dims, strides, box)) return kErrLaunch;
    if (encode_tmap_bf16_3d(&tv, c.v, dims, strides, box)) return kErrLaunch;
  }
  Params p;
  p.out = static_cast<__nv_bfloat16*>(c.out);
  p.T = c.T;
  p.start_pos = c.start_pos;
  p.H = c.H;
  p.Hkv = c.Hkv;
  p.group = group;
  p.tok_per_tile = tok_per_tile;
  p.window = c.window;
  p.units_per_head = (int)units;
  p.scale_log2 = (float)((double)c.scale * 1.4426950408889634);
  p.err = c.err;
  p.wait_limit_ns = c.wait_limit_ns;
  p.flags = c.flags;
  const dim3 grid((unsigned)(units * c.Hkv));
  if (p.scale_log2 > 0.f)
    bf16_d128_kernel<true><<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p);
  else
    bf16_d128_kernel<false><<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace pfa
