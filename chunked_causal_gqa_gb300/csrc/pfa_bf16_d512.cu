// pfa_bf16_d512.cu -- fused flash-style prefill attention for bf16, head_dim 512
// (the Gemma-style wide heads of the TensorSharp2 Gemma-4 prefill design,
// section 2: the head_dim-512 flash kernel, and its sliding-window layers),
// on the sm_103a tensor cores (tcgen05 + tensor memory + TMA), with the two
// CTAs of a cluster issuing their products together (cta_group::2).
//
// Operation: as for head_dim 128 (gnosis "Prefill attention -> GPU: handoff",
// section "GPU design", steps 1-3, fused).
//
// Budget that shapes this kernel: a 128 x 512 fp32 output accumulator would
// fill all 512 columns of tensor memory, leaving none for the scores, and one
// 128 x 512 bf16 query tile takes 128 KB of the 227 KB of shared memory.  So a
// CTA keeps one 128-row query tile (group heads x 128/group tokens) of one kv
// head and one half (256 columns) of the output head dimension, and another
// cluster computes the other half (both compute the full S = Q K^T: 1.5x the
// minimum tensor work, in exchange for fitting S and O in tensor memory).
//
// A 128-key tile needs the whole K tile (128 keys x 512) and the V rows of
// this output half: 192 KB, more than one SM takes in from L2 while its
// tensor core does the tile's 3k cycles of work.  So the two CTAs of a
// cluster (ranks 0 and 1, on two SMs) take query tiles 2p and 2p + 1 of the
// same kv head and output half, and rank 0 issues products of M = 256 rows
// for both (tcgen05.mma.cta_group::2): each CTA supplies its own 128 query
// rows (A) and half of the B operand -- keys 64 r .. 64 r + 63 of each K
// tile, output columns 128 r .. 128 r + 127 of this half of each V tile --
// and each CTA's tensor memory receives its own rows of S and O.  Every SM
// then takes in 96 KB per key tile.  The pair walks the union of its two
// tiles' key ranges; each CTA masks the keys its own rows do not see.
//
// Key tiles of 128: S products are M=256 N=128 K=16; the K slices stream
// through a ring of six 16 KB slots (two 64-key x 64-column boxes per slot,
// four slots per tile), this CTA's V slice as two slots (64 keys x 128
// columns each).  The producer of each CTA fills its ring in the order rank
// 0 consumes it: K(0), K(1), V(0), K(2), V(1), ...
//
// Warp roles (6 warps per CTA):
//   warps 0-3  softmax and epilogue (TMEM lanes 0-127, one row per thread)
//   warp  4    TMA producer: Q once, then this CTA's K and V slices.  The
//              loads of both CTAs complete on rank 0's barriers (TMA
//              .cta_group::2), so rank 0 sees when a slot is full in both.
//   warp  5    TMEM allocation (both ranks); on rank 0 the MMA issuer (one
//              elected lane issues each group of tcgen05.mma for the pair)
//
// Tensor memory (each CTA): [0,128) S_0, [128,256) S_1 (double-buffered
// scores; after the softmax the first 64 columns hold P as packed bf16
// pairs), [256,512) O half.
//
// MMA issue order: S(0), S(1), O += P(0) V(0), S(2), O += P(1) V(1), ...
// The softmax of tile i overlaps S(i+1); it waits for O += P(i-1) V(i-1)
// (barrier kBarO, one phase per tile) before it may rescale O.  Rank 0's
// commits arrive on the barrier at the same offset in both CTAs; rank 1's
// softmax warps arrive on rank 0's P barriers.
#include "pfa_internal.h"
#include "pfa_pair.cuh"
#include "pfa_ptx.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <vector>

namespace pfa {
namespace {

// ---------------------------------------------------------------- layout
constexpr int kBM = 128;                  // query rows per CTA (M = 256 per pair)
constexpr int kBN = 128;                  // keys per tile
constexpr int kKeysPerCta = 64;           // keys of each K tile in one CTA's slots
constexpr int kDHalf = 256;               // output columns per cluster
constexpr int kDQuarter = 128;            // V columns in one CTA's slots
constexpr int kQChunk = 128 * 128;        // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kSlot = 16384;              // ring slot: two 64 x 64 boxes
constexpr int kBox = 8192;                // 64 rows x 64 bf16
constexpr int kRing = 6;                  // ring slots
constexpr int kSmemQ = 0;                 // 8 chunks: 128 KB
constexpr int kSmemRing = 8 * kQChunk;    // 6 slots: 96 KB
constexpr int kSmemBars = kSmemRing + kRing * kSlot;  // 229376
constexpr int kSmemAlloc = kSmemBars + 256 + 1024;
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;

// Rank 0's kBarQ and kBarFull count the bytes of both CTAs' loads; rank 1's
// are unused.  kBarS, kBarO, kBarDrain and kBarEmpty receive rank 0's
// commits in both CTAs.
constexpr int kBarQ = 0;                  // both CTAs' Q have landed
constexpr int kBarS = 1;                  // 2
constexpr int kBarP = 3;                  // 2; rank 0: 8 arrivals (4 softmax warps per CTA)
constexpr int kBarO = 5;                  // one phase per tile's P V
constexpr int kBarDrain = 6;
constexpr int kBarFull = 7;               // kRing: the slot has landed in both CTAs
constexpr int kBarEmpty = kBarFull + kRing;  // kRing: the pair has consumed the slot
constexpr int kNumBars = kBarEmpty + kRing;
static_assert(kNumBars * 8 + 8 <= 256, "barrier area");
constexpr int kOffTmemSlot = kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;

constexpr uint32_t kColS = 0, kColO = 256;
constexpr uint32_t kIdescQK = idesc_bf16_f32(2 * kBM, kBN, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(2 * kBM, kDHalf, true);

// Tail split (with a caller workspace): the whole waves of units run whole;
// each unit of the last, partial wave is cut into `parts` equal key ranges
// run as separate clusters, part by part; a piece writes its unnormalised
// output halves, exponent bases and row sums to a workspace slot, and
// merge512_kernel combines the pieces of each unit in key order.
constexpr int kPlainMode = 0, kTailMode = 2;
constexpr size_t kOHalfFloats = (size_t)kBM * kDHalf;  // one CTA's O, [col/4][row][4]
// per piece: O for (rank, half) = 4 blocks, then base[4][128], sum[4][128]
constexpr size_t kPieceFloats = 4 * kOHalfFloats + 2 * 4 * kBM;

struct Params {
  __nv_bfloat16* out;
  float* ws;         // tail split: the pieces' slots; else null
  int mode, p1, p2, parts;
  int64_t o_stride;  // elements from one token's output row to the next
  int out_v8;        // output rows start on 32-byte boundaries
  int ring_rows;     // > 0: key j is in cache row j % ring_rows; 0: in row j
  int64_t T, start_pos;          // graph entry: T = the largest T, start_pos unused
  const int64_t* lens;           // graph entry: device {T, start_pos}; else null
  int64_t kv_capacity;           // rows per kv head in the cache
  int H, Hkv, group, tok_per_tile, window, tiles_per_head;
  float scale_log2;
  unsigned* err;
  uint64_t wait_limit_ns;
  int flags;
};

// Key tiles [first, first + n) of a unit: the union of the ranges of its two
// query tiles 2 pair and 2 pair + 1 (the second may lie past T).
struct UnitKeys {
  int64_t first;
  int n;
};
__host__ __device__ inline UnitKeys unit_keys(int64_t T, int64_t start_pos, int tok_per_tile,
                                              int window, int pair) {
  const int64_t t0a = (int64_t)(2 * pair) * tok_per_tile;
  int64_t t_end = t0a + 2 * (int64_t)tok_per_tile;
  if (t_end > T) t_end = T;
  const int64_t pos_first = start_pos + t0a;
  int64_t kmin = 0;
  if (window > 0 && pos_first - window + 1 > 0) kmin = pos_first - window + 1;
  UnitKeys u;
  u.first = kmin / kBN;
  u.n = (int)((start_pos + t_end - 1) / kBN - u.first + 1);
  return u;
}

template <bool kFoldScale, bool kDyn>
__global__ void __launch_bounds__(kThreads, 1)
bf16_d512_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
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
  const uint64_t lim = p.wait_limit_ns;
  const int rank = (int)cluster_ctarank();  // = blockIdx.x & 1 (clusters of two)

  // Chunk length and position: kernel parameters, or (graph entry, kDyn) read
  // from device memory at run time, with the grid sized for the largest T.
  // Both CTAs of a cluster take every decision below from the same values.
  int64_t T = p.T, start_pos = p.start_pos;
  int tiles_per_head = p.tiles_per_head;
  if (kDyn) {
    T = p.lens[0];
    start_pos = p.lens[1];
    if (!lengths_ok(T, start_pos, p.T, p.kv_capacity, p.ring_rows, p.window)) {
      if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, kErrLengths);
      return;
    }
    tiles_per_head = (int)((T + p.tok_per_tile - 1) / p.tok_per_tile);
    if ((int)(blockIdx.x >> 2) >= ((tiles_per_head + 1) / 2) * p.Hkv) return;  // nothing set up yet
  }
  const int npairs = (tiles_per_head + 1) / 2;

  // Cluster c = blockIdx.x / 2 computes output half dh = c % 2 of unit c / 2,
  // or, past the whole waves of a tail split, part r of unit p1 + e.
  // Unit: (kv head, pair of query tiles); latest tokens first.
  const int cl = (int)(blockIdx.x >> 1);
  const int dh = cl & 1;
  const int pidx = cl >> 1;
  int rest = pidx, part = 0, slot = -1;
  if (p.mode == kTailMode && pidx >= p.p1) {
    const int j = pidx - p.p1;
    part = j / p.p2;
    rest = p.p1 + j % p.p2;
    slot = j;
  }
  const int kh = rest % p.Hkv;
  const int pair = npairs - 1 - rest / p.Hkv;
  const int tile = 2 * pair + rank;
  const int64_t t0 = (int64_t)tile * p.tok_per_tile;
  const int64_t pos_first = start_pos + t0;
  const int64_t pos_last = start_pos + t0 + p.tok_per_tile - 1;
  const UnitKeys uk = unit_keys(T, start_pos, p.tok_per_tile, p.window, pair);
  const int kb = slot < 0 ? 0 : (int)((int64_t)uk.n * part / p.parts);
  const int ke = slot < 0 ? uk.n : (int)((int64_t)uk.n * (part + 1) / p.parts);
  const int64_t kt_first = uk.first + kb;  // first key tile of this cluster's range
  const int n = ke - kb;
  auto key_row = [&](int64_t key) -> int {
    return (int)(p.ring_rows > 0 ? key % p.ring_rows : key);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(bar(i), (i == kBarP || i == kBarP + 1) ? 8u : 1u);  // P: one arrival per softmax warp of the pair
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Ring order (producers and consumer): for i = 0..n-1: the four K slots of
  // tile i, then (i >= 1) the two V slots of tile i-1; after the last tile,
  // the V slots of tile n-1.  Six loads per tile.

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int hq = kh * p.group;
      // rank 0 arms its barrier for the bytes of both CTAs; rank 1's bytes
      // may land first (the phase cannot complete before rank 0's arrival)
      const uint32_t bar0 = cluster_addr(bar(0), 0);  // rank 0's barrier area
      auto bar_r0 = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
      if (rank == 0)
        mbar_arrive_expect_tx(bar(kBarQ), 2u * 8u * 128u * (uint32_t)(p.group * p.tok_per_tile));
      for (int c = 0; c < 8; ++c)
        tma_load_3d_pair(sbase + kSmemQ + c * kQChunk, &tm_q, bar_r0(kBarQ), 64 * c, hq, (int)t0);
      uint32_t li = 0;  // slot loads issued
      bool ok = true;
      auto slot_wait = [&](uint32_t* dst) -> bool {
        const uint32_t s = li % kRing, ph = (li / kRing) & 1u;
        if (!mbar_wait(bar(kBarEmpty + s), ph ^ 1u, abort_flag, p.err, lim)) return false;
        if (rank == 0) mbar_arrive_expect_tx(bar(kBarFull + s), 2u * (uint32_t)kSlot);
        *dst = s;
        return true;
      };
      auto load_k = [&](int i) -> bool {  // keys 64 rank .. +63 of tile i, all 512 columns
        const int row = key_row((kt_first + i) * kBN + kKeysPerCta * rank);
        for (int c = 0; c < 4; ++c) {
          uint32_t s;
          if (!slot_wait(&s)) return false;
          for (int b = 0; b < 2; ++b)
            tma_load_3d_pair(sbase + kSmemRing + s * kSlot + b * kBox, &tm_k, bar_r0(kBarFull + s),
                             128 * c + 64 * b, row, kh);
          ++li;
        }
        return true;
      };
      auto load_v = [&](int i) -> bool {  // columns 128 rank .. +127 of this half
        const int col = dh * kDHalf + kDQuarter * rank;
        for (int h = 0; h < 2; ++h) {
          const int row = key_row((kt_first + i) * kBN + kKeysPerCta * h);
          uint32_t s;
          if (!slot_wait(&s)) return false;
          for (int b = 0; b < 2; ++b)
            tma_load_3d_pair(sbase + kSmemRing + s * kSlot + b * kBox, &tm_v, bar_r0(kBarFull + s),
                             col + 64 * b, row, kh);
          ++li;
        }
        return true;
      };
      for (int i = 0; i < n && ok; ++i) {
        ok = load_k(i);
        if (ok && i > 0) ok = load_v(i - 1);
      }
      if (ok) ok = load_v(n - 1);
      // No copy may be in flight when either CTA exits: rank 0 waits for the
      // last loads of both (its barriers count both CTAs' bytes) before the
      // final cluster barrier.  On the normal path the pair has already
      // consumed every load, so these return at once.
      if (rank == 0) {
        mbar_wait(bar(kBarQ), 0, abort_flag, p.err, lim, true);
        const uint32_t first = li > (uint32_t)kRing ? li - kRing : 0;
        for (uint32_t j = first; j < li; ++j)
          mbar_wait(bar(kBarFull + j % kRing), (j / kRing) & 1u, abort_flag, p.err, lim, true);
      }
    }
  } else if (warp == 5 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    // The whole warp runs this loop (operands stay warp-uniform); one elected
    // lane issues each group of MMAs and each commit.
    {
      const uint32_t tO = tmem + kColO;
      bool ok = mbar_wait_warp(bar(kBarQ), 0, abort_flag, p.err, lim);
      tc_fence_after();
      bool issued = false;
      uint32_t li = 0;  // slot loads consumed
      auto slot_ready = [&](uint32_t* s) -> bool {
        *s = li % kRing;
        if (!mbar_wait_warp(bar(kBarFull + *s), (li / kRing) & 1u, abort_flag, p.err, lim))
          return false;
        tc_fence_after();
        return true;
      };
      auto pv = [&](int j) -> bool {  // O (+)= P(j) V(j)
        if (!mbar_wait_cl_warp(bar(kBarP + (j & 1)), (uint32_t)(j >> 1) & 1u, abort_flag, p.err,
                               lim))
          return false;
        tc_fence_after();
        const uint32_t tP = tmem + kColS + (uint32_t)((j & 1) * kBN);
        for (int h = 0; h < 2; ++h) {
          uint32_t s;
          if (!slot_ready(&s)) return false;
          ++li;
          // 64 keys = 4 steps of 16 (2048 B apart); each CTA's 128 columns are
          // two 64-column boxes (LBO = one box, 8 KB)
          mma4_ts_pair<2048 / 16>(tO, tP + 32u * h, sdesc_sw128(sbase + kSmemRing + s * kSlot, kBox, 1024),
                                  kIdescPV, (j > 0 || h > 0) ? 1u : 0u);
          tc_commit_pair(bar(kBarEmpty + s));
        }
        tc_commit_pair(bar(kBarO));
        return true;
      };
      for (int i = 0; i < n && ok; ++i) {
        const uint32_t tS = tmem + kColS + (uint32_t)((i & 1) * kBN);
#pragma unroll 1
        for (int c = 0; c < 4 && ok; ++c) {
          uint32_t s;
          if (!(ok = slot_ready(&s))) break;
          // Q columns 128 c .. 128 c + 127 (chunks 2c, 2c + 1) against the two
          // 64-column boxes of the slot
          mma8_ss_pair<kQChunk / 16, kBox / 16>(
              tS, sdesc_sw128(sbase + kSmemQ + 2 * c * kQChunk, 16, 1024),
              sdesc_sw128(sbase + kSmemRing + s * kSlot, 16, 1024), kIdescQK, c > 0 ? 1u : 0u);
          issued = true;
          tc_commit_pair(bar(kBarEmpty + s));
          ++li;
        }
        if (!ok) break;
        tc_commit_pair(bar(kBarS + (i & 1)));
        if (i > 0 && !(ok = pv(i - 1))) break;
      }
      if (ok) ok = pv(n - 1);
      if (issued) {
        tc_commit_pair(bar(kBarDrain));
        mbar_wait_warp(bar(kBarDrain), 0, abort_flag, p.err, lim, true);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int row = warp * 32 + lane;
    const int tok = row / p.group;
    const bool row_exists = tok < p.tok_per_tile;
    const int64_t t = t0 + tok;
    const bool row_valid = row_exists && t < T;
    const int64_t pos = start_pos + t;
    const int h = kh * p.group + row % p.group;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + lane_off + kColO;
    const float c = p.scale_log2;
    const uint32_t bar_p[2] = {cluster_addr(bar(kBarP), 0), cluster_addr(bar(kBarP + 1), 0)};  // rank 0's

    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    if (p.flags & kFlagForceTimeout) {
      ok = mbar_wait(bar(kBarDrain), 0, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    for (int i = 0; i < n && ok; ++i) {
      ok = mbar_wait(bar(kBarS + (i & 1)), (uint32_t)(i >> 1) & 1u, abort_flag, p.err, lim);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + kColS + (uint32_t)((i & 1) * kBN);
      uint32_t r0[32], r1[32], r2[32], r3[32];  // four loads in flight
      tmem_ld32(tS, r0);
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
      const int64_t key0 = (kt_first + i) * kBN;
      const bool all_visible = (key0 + kBN - 1 <= pos_first) &&
                               (p.window <= 0 || key0 > pos_last - p.window);
      if (!all_visible) {
        const int64_t hi = pos - key0;
        const int64_t lo = p.window > 0 ? pos - p.window - key0 : -1;
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j > hi || j <= lo) x[j] = -INFINITY;
      }
      // row max with three-input max instructions in 8 independent chains
      float mx;
      {
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
      if (kFoldScale) mx *= c;
      float alpha = 1.f;
      bool rescale = false;
      if (mx > m_run + kRescaleThreshold) {
        alpha = ex2(m_run - mx);
        rescale = (i > 0) && (m_run != -INFINITY);
        m_run = mx;
      }
      const float base = (m_run == -INFINITY) ? 0.f : m_run;
      // P = 2^(s - base) as packed bf16 pairs; l gains the row sum of the
      // unrounded values (8 independent partial sums)
      uint32_t pk0[32], pk1[32];
      float ls[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) ls[q] = 0.f;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float xa = x[2 * j], xb = x[2 * j + 1];
        const float pa = kFoldScale ? ex2(fmaf(xa, c, -base)) : ex2(xa - base);
        const float pb = kFoldScale ? ex2(fmaf(xb, c, -base)) : ex2(xb - base);
        const uint32_t w = pack_bf16x2(pa, pb);
        if (j < 32) pk0[j] = w; else pk1[j - 32] = w;
        ls[(2 * j) & 7] += pa;
        ls[(2 * j + 1) & 7] += pb;
      }
      const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      l = l * alpha + lsum;
      if (i > 0) {
        // O (and the P buffer this tile reuses) are free once P(i-1) V is done.
        ok = mbar_wait(bar(kBarO), (uint32_t)(i - 1) & 1u, abort_flag, p.err, lim);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < kDHalf; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st32(tO + c0, o);
        }
      }
      tmem_st32(tS, pk0);
      tmem_st32(tS + 32, pk1);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(bar_p[i & 1]);
    }
    if (ok) {
      ok = mbar_wait(bar(kBarO), (uint32_t)(n - 1) & 1u, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok && slot >= 0) {
      // piece of a split unit: unnormalised fp32 output half, base and sum
      tc_fence_after();
      const int blk = rank * 2 + dh;
      float* ws = p.ws + (size_t)slot * kPieceFloats;
      float4* ocol = reinterpret_cast<float4*>(ws + (size_t)blk * kOHalfFloats) + row;
#pragma unroll 1
      for (int c0 = 0; c0 < kDHalf; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c0, o);
        tmem_wait_ld(o);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          ocol[(size_t)(c0 / 4 + j) * kBM] =
              make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                          __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
      }
      ws[4 * kOHalfFloats + blk * kBM + row] = m_run;
      ws[4 * kOHalfFloats + 4 * kBM + blk * kBM + row] = l;
    } else if (ok) {
      tc_fence_after();
      // Each thread writes its row's 512 contiguous bytes: with 32-byte
      // aligned rows, in 32-byte stores (whole L2 sectors; measured 57.7 ->
      // 55.6 us on the window layer against 16-byte stores).
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.out + (t * p.o_stride + h * (int64_t)512 + dh * kDHalf);
#pragma unroll 1
      for (int c0 = 0; c0 < kDHalf; c0 += 64) {
        uint32_t o[32], o2[32];
        tmem_ld32(tO + c0, o);
        tmem_ld32(tO + c0 + 32, o2);
        tmem_wait_ld(o);
        tmem_wait_ld(o2);
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
          w[16 + j] = pack_bf16x2(__uint_as_float(o2[2 * j]) * inv, __uint_as_float(o2[2 * j + 1]) * inv);
        }
        if (row_valid) {
          if (p.out_v8) {
#pragma unroll
            for (int j = 0; j < 4; ++j) st_global_v8(orow + c0 + 16 * j, &w[8 * j]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          }
        }
      }
    }
  }

  // Neither CTA leaves, nor frees tensor memory, while the pair's products
  // or copies may still touch it: rank 0 drains both before this point.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Combines the pieces of each split unit in key order:
// m = max_r m_r, O = sum_r 2^(m_r - m) O_r, l = sum_r 2^(m_r - m) l_r, out = O / l.
// Block (e, g, rank): query tile 2 pair + rank of unit p1 + e, output columns
// 16 g .. 16 g + 15; thread = row (the pieces' [col/4][row][4] layout makes
// every load coalesced).
constexpr int kMerge512Cols = 16;

__global__ void __launch_bounds__(kBM) merge512_kernel(const Params p) {
  const int e = blockIdx.x;
  const int unit = p.p1 + e;
  const int rank = blockIdx.z;
  const int kh = unit % p.Hkv;
  const int npairs = (p.tiles_per_head + 1) / 2;
  const int tile = 2 * (npairs - 1 - unit / p.Hkv) + rank;
  const int row = threadIdx.x;
  const int tok = row / p.group;
  const int64_t t = (int64_t)tile * p.tok_per_tile + tok;
  if (tok >= p.tok_per_tile || t >= p.T) return;
  const int h = kh * p.group + row % p.group;
  const int col0 = blockIdx.y * kMerge512Cols;
  const int dh = col0 / kDHalf;
  const int blk = rank * 2 + dh;
  const int cq0 = (col0 % kDHalf) / 4;  // first column quad within the half
  auto piece = [&](int r) -> const float* {
    return p.ws + (size_t)(r * p.p2 + e) * kPieceFloats;
  };
  const size_t off_m = 4 * kOHalfFloats + (size_t)blk * kBM + row, off_l = off_m + 4 * kBM;
  float m = -INFINITY;
  for (int r = 0; r < p.parts; ++r) m = fmaxf(m, piece(r)[off_m]);
  const float mb = (m == -INFINITY) ? 0.f : m;
  float4 acc[kMerge512Cols / 4];
#pragma unroll
  for (int q = 0; q < kMerge512Cols / 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  for (int r = 0; r < p.parts; ++r) {
    const float* ws = piece(r);
    const float w = ex2(ws[off_m] - mb);  // 0 for a piece that saw no visible key
    l = fmaf(w, ws[off_l], l);
    const float4* ocol = reinterpret_cast<const float4*>(ws + (size_t)blk * kOHalfFloats) + row;
#pragma unroll
    for (int q = 0; q < kMerge512Cols / 4; ++q) {
      const float4 o = ocol[(size_t)(cq0 + q) * kBM];
      acc[q].x = fmaf(w, o.x, acc[q].x);
      acc[q].y = fmaf(w, o.y, acc[q].y);
      acc[q].z = fmaf(w, o.z, acc[q].z);
      acc[q].w = fmaf(w, o.w, acc[q].w);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint32_t wv[kMerge512Cols / 2];
#pragma unroll
  for (int q = 0; q < kMerge512Cols / 4; ++q) {
    wv[2 * q] = pack_bf16x2(acc[q].x * inv, acc[q].y * inv);
    wv[2 * q + 1] = pack_bf16x2(acc[q].z * inv, acc[q].w * inv);
  }
  uint4* dst = reinterpret_cast<uint4*>(p.out + t * p.o_stride + h * (int64_t)512 + col0);
#pragma unroll
  for (int q = 0; q < kMerge512Cols / 8; ++q)
    dst[q] = make_uint4(wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
}

// ------------------------------------------------------------------ host
// Schedule of one shape: plain, or the tail split.
struct Plan512 {
  int mode = kPlainMode, p1 = 0, p2 = 0, parts = 0;
  size_t ws_bytes = 0;
};

// Fixed cost of a cluster (Q load, pipeline fill, epilogue) and of the
// merge, in key-tile units.
constexpr int64_t kCtaOverheadTiles = 2, kMerge512CostTiles = 2;
constexpr int kMaxParts512 = 8;

// Makespan, in key-tile units, of clusters launched in order on `slots`
// pairs of SMs (the hardware starts each on the first pair that frees up).
int64_t makespan(const std::vector<int64_t>& costs, int slots) {
  std::vector<int64_t> free_at((size_t)std::max(slots, 1), 0);
  int64_t end = 0;
  for (int64_t cost : costs) {
    std::pop_heap(free_at.begin(), free_at.end(), std::greater<int64_t>());
    free_at.back() += cost;
    end = std::max(end, free_at.back());
    std::push_heap(free_at.begin(), free_at.end(), std::greater<int64_t>());
  }
  return end;
}

// The tail split is taken when it beats the plain schedule's estimate by 5%.
// Units (kv head, pair of query tiles) take four CTAs: two clusters, one per
// output half.
Plan512 plan_d512(const Call& c) {
  Plan512 plan;
  if (c.lens != nullptr || c.num_sms < 4) return plan;
  const int group = c.H / c.Hkv;
  const int tok_per_tile = kBM / group;
  const int64_t tiles = (c.T + tok_per_tile - 1) / tok_per_tile;
  const int64_t npairs = (tiles + 1) / 2;
  const int64_t U = npairs * c.Hkv;
  const int per_wave = c.num_sms / 4;  // units per wave
  const int slots = c.num_sms / 2;     // clusters in flight
  if (U <= per_wave || U > (1 << 20)) return plan;
  const int p1 = per_wave * (int)(U / per_wave), p2 = (int)(U - p1);
  if (p2 == 0) return plan;
  std::vector<int> n((size_t)U);
  int nmin = INT32_MAX;
  for (int u = 0; u < (int)U; ++u) {
    const int pair = (int)npairs - 1 - u / c.Hkv;
    n[u] = unit_keys(c.T, c.start_pos, tok_per_tile, c.window, pair).n;
    if (u >= p1) nmin = std::min(nmin, n[u]);
  }
  std::vector<int64_t> costs;
  for (int u = 0; u < (int)U; ++u)
    for (int d = 0; d < 2; ++d) costs.push_back(n[u] + kCtaOverheadTiles);
  const int64_t plain = makespan(costs, slots);
  int64_t best = INT64_MAX;
  for (int parts = 2; parts <= kMaxParts512 && parts <= nmin; ++parts) {
    costs.clear();
    for (int u = 0; u < p1; ++u)
      for (int d = 0; d < 2; ++d) costs.push_back(n[u] + kCtaOverheadTiles);
    for (int r = 0; r < parts; ++r)
      for (int e = 0; e < p2; ++e) {
        const int64_t nu = n[p1 + e];
        for (int d = 0; d < 2; ++d)
          costs.push_back(nu * (r + 1) / parts - nu * r / parts + kCtaOverheadTiles);
      }
    const int64_t m = makespan(costs, slots) + kMerge512CostTiles;
    if (m < best) {
      best = m;
      plan.parts = parts;
    }
  }
  if (plan.parts == 0 || best * 100 >= plain * 95) return Plan512{};
  plan.mode = kTailMode;
  plan.p1 = p1;
  plan.p2 = p2;
  plan.ws_bytes = (size_t)p2 * plan.parts * kPieceFloats * sizeof(float);
  return plan;
}

}  // namespace

// Host replay of the work assignment of a launch (schedule of `c` on `sms`
// SMs): the kernel's CTA -> (cluster, rank, item) mapping, run for every CTA
// of the grid, and the merge's reads.  Returns 0, or the number of the first
// failed check.
int check_schedule_bf16_d512(const Call& c0, int sms, int* schedule, int* ctas) {
  Call c = c0;
  c.num_sms = sms;
  c.lens = nullptr;
  const Plan512 plan = plan_d512(c);
  *schedule = plan.mode == kTailMode ? 2 : 0;
  const int group = c.H / c.Hkv;
  const int tok_per_tile = kBM / group;
  const int64_t tiles = (c.T + tok_per_tile - 1) / tok_per_tile;
  const int npairs = (int)((tiles + 1) / 2);
  const int64_t units = plan.mode == kTailMode ? (int64_t)plan.p1 + (int64_t)plan.p2 * plan.parts
                                               : (int64_t)npairs * c.Hkv;
  const int64_t grid = 4 * units;
  if (grid > (1 << 24)) return 1;
  *ctas = (int)grid;
  const int64_t L = c.start_pos + c.T;
  const int pieces = plan.mode == kTailMode ? plan.p2 * plan.parts : 0;
  struct Cover {
    int64_t kb, ke;
    int slot;
  };
  std::vector<std::vector<Cover>> cover((size_t)(c.Hkv * tiles * 2));
  std::vector<int> slot_ctas((size_t)pieces, 0);
  for (int64_t b = 0; b < grid; ++b) {
    const int rank = (int)(b & 1), cl = (int)(b >> 1), dh = cl & 1, pidx = cl >> 1;
    int rest = pidx, part = 0, slot = -1;
    if (plan.mode == kTailMode && pidx >= plan.p1) {
      const int j = pidx - plan.p1;
      part = j / plan.p2;
      rest = plan.p1 + j % plan.p2;
      slot = j;
    }
    const int kh = rest % c.Hkv;
    const int pair = npairs - 1 - rest / c.Hkv;
    if (kh < 0 || kh >= c.Hkv || pair < 0 || pair >= npairs) return 2;
    const UnitKeys uk = unit_keys(c.T, c.start_pos, tok_per_tile, c.window, pair);
    const int kb = slot < 0 ? 0 : (int)((int64_t)uk.n * part / plan.parts);
    const int ke = slot < 0 ? uk.n : (int)((int64_t)uk.n * (part + 1) / plan.parts);
    if (uk.n < 1 || ke <= kb) return 3;                       // every cluster walks a key tile
    if (uk.first < 0 || (uk.first + uk.n - 1) * kBN > L - 1) return 4;  // tiles start inside the cache
    // TMA x coordinates of the 64-column boxes: Q and K at 64 q, V at this
    // CTA's columns of the half: 16-byte aligned and inside the 512 columns
    for (int q = 0; q < 8; ++q)
      if ((64 * q) % 8 || 64 * q + 64 > 512) return 5;
    for (int bb = 0; bb < 2; ++bb) {
      const int x = dh * kDHalf + kDQuarter * rank + 64 * bb;
      if (x % 8 || x + 64 > 512) return 5;
    }
    const int tile = 2 * pair + rank;
    const int64_t t0 = (int64_t)tile * tok_per_tile;
    if (t0 >= c.T) {
      if (tile != tiles || rank != 1) return 6;  // only the second tile of an odd last pair
      continue;
    }
    for (int64_t t = t0; t < t0 + tok_per_tile && t < c.T; ++t) {
      const int64_t pos = c.start_pos + t;
      const int64_t lo = c.window > 0 ? std::max<int64_t>(0, pos - c.window + 1) : 0;
      if (lo < uk.first * kBN || pos >= (uk.first + uk.n) * kBN) return 7;  // visible keys walked
    }
    if (slot >= 0) {
      if (slot >= pieces) return 8;
      ++slot_ctas[(size_t)slot];
    }
    cover[(size_t)((kh * tiles + tile) * 2 + dh)].push_back({uk.first + kb, uk.first + ke, slot});
  }
  for (int j = 0; j < pieces; ++j)
    if (slot_ctas[(size_t)j] != 4) return 9;  // a piece slot: both ranks, both halves
  for (int kh = 0; kh < c.Hkv; ++kh)
    for (int64_t tile = 0; tile < tiles; ++tile) {
      const int pair = (int)(tile / 2);
      const UnitKeys uk = unit_keys(c.T, c.start_pos, tok_per_tile, c.window, pair);
      const int unit = (npairs - 1 - pair) * c.Hkv + kh;
      const bool split = plan.mode == kTailMode && unit >= plan.p1;
      for (int dh = 0; dh < 2; ++dh) {
        std::vector<Cover> v = cover[(size_t)((kh * tiles + tile) * 2 + dh)];
        std::sort(v.begin(), v.end(), [](const Cover& a, const Cover& b) { return a.kb < b.kb; });
        if (!split) {
          // one whole item writes the output
          if (v.size() != 1 || v[0].slot >= 0 || v[0].kb != uk.first || v[0].ke != uk.first + uk.n)
            return 10;
          continue;
        }
        // the pieces cover the unit's key tiles in order, and the merge of
        // unit p1 + e reads exactly their slots r * p2 + e, r = 0 .. parts-1
        if ((int)v.size() != plan.parts) return 11;
        const int e = unit - plan.p1;
        int64_t at = uk.first;
        for (int r = 0; r < plan.parts; ++r) {
          if (v[(size_t)r].kb != at || v[(size_t)r].slot != r * plan.p2 + e) return 12;
          at = v[(size_t)r].ke;
        }
        if (at != uk.first + uk.n) return 13;
      }
    }
  if (plan.mode == kTailMode && plan.ws_bytes < (size_t)pieces * kPieceFloats * sizeof(float))
    return 14;
  return 0;
}

size_t workspace_bytes_bf16_d512(const Call& c, int* schedule) {
  const Plan512 plan = plan_d512(c);
  if (schedule) *schedule = plan.mode == kTailMode ? 2 : 0;
  return plan.ws_bytes;
}

int launch_bf16_d512(const Call& c) {
  static DeviceOnce setup;
  const int sr = setup.run(c.device, [] {
    const void* fns[4] = {(const void*)bf16_d512_kernel<true, false>,
                          (const void*)bf16_d512_kernel<false, false>,
                          (const void*)bf16_d512_kernel<true, true>,
                          (const void*)bf16_d512_kernel<false, true>};
    for (const void* fn : fns)
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) !=
          cudaSuccess)
        return kErrLaunch;
    return kOk;
  });
  if (sr != kOk) return sr;
  const int group = c.H / c.Hkv;
  const int tok_per_tile = kBM / group;
  const int64_t tiles = (c.T + tok_per_tile - 1) / tok_per_tile;
  const int64_t npairs = (tiles + 1) / 2;
  const int64_t L = c.start_pos + c.T;
  if (4 * npairs * c.Hkv > 0x7fffffff || L + 2 * kBN > 0x7fffffff) return kErrShape;

  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {512, (uint64_t)c.H, (uint64_t)c.T};
    const uint64_t strides[2] = {512 * 2, (uint64_t)c.qkv_dim * 2};
    const uint32_t box[3] = {64, (uint32_t)group, (uint32_t)tok_per_tile};
    if (encode_tmap_bf16_3d(&tq, c.q, dims, strides, box)) return kErrLaunch;
  }
  {
    // Rows past the written part of the cache read as zeros.  K and V move
    // in boxes of 64 keys x 64 columns.
    const uint64_t dims[3] = {512, (uint64_t)cache_rows_written(c), (uint64_t)c.Hkv};
    const uint64_t strides[2] = {512 * 2, (uint64_t)c.max_seq_len * 512 * 2};
    const uint32_t box[3] = {64, (uint32_t)kKeysPerCta, 1};
    if (encode_tmap_bf16_3d(&tk, c.k, dims, strides, box)) return kErrLaunch;
    if (encode_tmap_bf16_3d(&tv, c.v, dims, strides, box)) return kErrLaunch;
  }
  // the tail split when the caller gave a large enough workspace
  Plan512 plan;
  if (c.ws != nullptr && c.lens == nullptr) {
    plan = plan_d512(c);
    if (plan.ws_bytes > c.ws_bytes) plan = Plan512{};
  }
  Params p;
  p.out = static_cast<__nv_bfloat16*>(c.out);
  p.ws = plan.mode == kTailMode ? static_cast<float*>(c.ws) : nullptr;
  p.mode = plan.mode;
  p.p1 = plan.p1;
  p.p2 = plan.p2;
  p.parts = plan.parts;
  p.o_stride = c.qkv_dim;
  p.out_v8 = (reinterpret_cast<uintptr_t>(c.out) % 32 == 0 && c.qkv_dim % 16 == 0) ? 1 : 0;
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
  const int64_t units = plan.mode == kTailMode
                            ? (int64_t)plan.p1 + (int64_t)plan.p2 * plan.parts
                            : npairs * c.Hkv;
  // Clusters of two consecutive CTAs: the two query tiles of a unit, for one
  // output half.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(4 * units));
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
  const bool fold = p.scale_log2 > 0.f;
  cudaError_t e;
  if (c.lens)
    e = fold ? cudaLaunchKernelEx(&cfg, bf16_d512_kernel<true, true>, tq, tk, tv, p)
             : cudaLaunchKernelEx(&cfg, bf16_d512_kernel<false, true>, tq, tk, tv, p);
  else
    e = fold ? cudaLaunchKernelEx(&cfg, bf16_d512_kernel<true, false>, tq, tk, tv, p)
             : cudaLaunchKernelEx(&cfg, bf16_d512_kernel<false, false>, tq, tk, tv, p);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return kErrLaunch;
  if (plan.mode == kTailMode) {
    merge512_kernel<<<dim3((unsigned)plan.p2, 512 / kMerge512Cols, 2), kBM, 0, c.stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
  }
  return kOk;
}

}  // namespace pfa
