// pfa_bf16_d128.cu -- fused flash-style prefill attention for bf16, head_dim 128,
// on the sm_103a tensor cores (tcgen05 + tensor memory + TMA).
//
// Operation (gnosis "Prefill attention -> GPU: handoff", section "GPU design",
// steps 1-3, fused): per query row, scores against the visible keys of its kv
// head, scale, causal (+ window) mask, softmax, weighted sum of V.
//
// Pair (the unit of query work): one kv head and two consecutive 128-row query
// tiles, A and B.  A tile packs all `group` query heads of the kv head for
// 128 / group consecutive tokens (row r -> token r / group, head r % group),
// so every K/V tile that TMA brings into shared memory feeds all heads of the
// GQA group, and both tiles.
//
// Work item: a pair and a range [kb, ke) of its key tiles.  A CTA executes a
// list of items in order.  With the plain schedule every CTA runs one item,
// a whole pair, and writes the normalised output.  Two schedules need a
// caller-provided workspace; an item that covers only part of a pair writes
// its unnormalised partial (O, exponent base, row sum) to a workspace slot,
// and merge_kernel combines the pieces of each such pair in a fixed order
// (the log-sum-exp identity of the softmax; the result is deterministic):
//   * tail split: with more pairs than SMs, the whole waves run whole and
//     each pair of the last, partial wave is cut into equal key ranges, so
//     the last wave fills the SMs (long chunks deep in a context); with no
//     more pairs than SMs, every pair is cut the same way in one wave (short
//     chunks deep in a context: the CTAs of one range share its keys in L2);
//   * balanced: the host cuts the pairs' key tiles into at most one run of
//     items per SM, of equal cost (tiles plus a fixed per-item overhead) --
//     chiefly short chunks deep into long contexts, where the plain schedule
//     has fewer pairs than SMs.
// The host picks a workspace schedule only where its estimated makespan
// beats the plain one's by a margin.
//
// Warp roles (10 warps):
//   warps 0-3  softmax for tile A (TMEM lanes 0-127, one row per thread)
//   warps 4-7  softmax for tile B
//   warp  8    TMA producer: Q tiles of each item, K/V tiles into a 5-slot ring
//   warp  9    TMEM allocator and MMA issuer.  The whole warp runs the issue
//              loop, so the operand descriptors stay warp-uniform, and one
//              elected lane issues each group of eight tcgen05.mma.  (Issuing
//              from a lone lane of a diverged warp costs ~90 cycles per MMA,
//              more than the 64 cycles an M=128 N=128 K=16 product takes.)
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
// normalisation O / l is exact for any base.  l is summed from the fp32
// probabilities before their rounding to bf16 for the P V product.
//
// Masks come from indices: key j is visible to a row at position pos iff
// j <= pos and (window <= 0 or j > pos - window).  Key tiles outside every
// row's band are never loaded; tiles fully inside every row's band skip the
// per-element test.
//
// Registers: 10 warps put three warps on some of the SM's four register-file
// partitions, which caps a thread at 168 registers.
#include "pfa_internal.h"
#include "pfa_ptx.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <memory>
#include <mutex>
#include <vector>

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
constexpr int kBarQFree = 1;                 // Q buffers no longer read by the item's MMAs
constexpr int kBarFull = 2;                  // kSlots
constexpr int kBarEmpty = kBarFull + kSlots; // kSlots
constexpr int kBarS = kBarEmpty + kSlots;    // 2 (A, B)
constexpr int kBarP = kBarS + 2;             // 2
constexpr int kBarO = kBarP + 2;             // 2: item's accumulators complete
constexpr int kBarOFree = kBarO + 2;         // 2: item's epilogue has read O
constexpr int kBarDrain = kBarOFree + 2;
constexpr int kBarQB = kBarDrain + 1;        // short launches: Q_B loaded (kBarQ then covers Q_A)
constexpr int kNumBars = kBarQB + 1;
constexpr int kOffTmemSlot = kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
static_assert(kOffAbort + 4 <= 256, "barrier area");

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false);  // K-major Q and K
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, 128, true);   // V is N(=d)-contiguous

// ---- schedule tables (kernel parameters)
constexpr int kMaxCtas = 192;
constexpr int kMaxItems = 512;
constexpr int kMaxMerge = 256;
constexpr int kMaxPieces = 512;
constexpr int kPairRows = 2 * kBM;
constexpr size_t kSlotFloats = (size_t)kPairRows * 128 + 2 * kPairRows;  // O, base, sum
constexpr size_t kSlotBytes = kSlotFloats * sizeof(float);

struct Item {
  int pair, kb, ke, slot;  // key tiles [kb, ke) of the pair; slot < 0: whole pair, direct output
};
// Schedule modes.
//   kPlain:  CTA b runs pair b whole.
//   kTable:  CTA c runs items [cta_first[c], cta_first[c+1]) of `items`.
//   kTail:   CTAs 0 .. p1-1 run pairs 0 .. p1-1 whole; then, part by part,
//            CTA p1 + r * p2 + e runs part r (of `parts` equal key ranges) of
//            pair p1 + e into workspace slot r * p2 + e.
constexpr int kPlain = 0, kTable = 1, kTail = 2;
// Plain launches whose longest pair holds at most this many key tiles take
// the short-launch kernel variant (kShort).
constexpr int kShortTiles = 64;
struct Sched {
  int mode;
  int p1, p2, parts;
  int cta_first[kMaxCtas + 1];
  Item items[kMaxItems];
};
// The plain and tail-split modes need only the head of the schedule.  Their
// kernels take this 16-byte block instead of the ~9 KB table: the large
// parameter block costs launch time, and the table code left the hot loop
// short of registers (spills).
struct SchedLite {
  int mode;
  int p1, p2, parts;
};
__device__ __forceinline__ int table_first(const Sched& s, int c) { return s.cta_first[c]; }
__device__ __forceinline__ int table_first(const SchedLite&, int) { return 0; }
__device__ __forceinline__ Item table_item(const Sched& s, int k) { return s.items[k]; }
__device__ __forceinline__ Item table_item(const SchedLite&, int) { return Item{0, 0, 0, -1}; }
struct MergeEntry {
  int pair, first, count, pad;  // pieces slots[first .. first+count), in key order
};
struct MergeSched {
  int num;     // entries (tail layout: the p2 tail pairs, entry e -> pair p1 + e)
  int tail;    // 1: entries follow the kTail layout; e and slots are unused
  int p1, p2, parts;
  MergeEntry e[kMaxMerge];
  int slots[kMaxPieces];
};

// The tail-split merge needs only the head.
struct MergeLite {
  int num, tail, p1, p2, parts;
};
__device__ __forceinline__ MergeEntry merge_entry(const MergeSched& ms, int b) { return ms.e[b]; }
__device__ __forceinline__ MergeEntry merge_entry(const MergeLite&, int) {
  return MergeEntry{0, 0, 0, 0};
}
__device__ __forceinline__ int merge_slot(const MergeSched& ms, int i) { return ms.slots[i]; }
__device__ __forceinline__ int merge_slot(const MergeLite&, int) { return 0; }

struct Params {
  __nv_bfloat16* out;
  float* ws;  // partial slots (balanced schedule only)
  int64_t o_stride;  // elements from one token's output row to the next
  int ring_rows;     // > 0: key j is in cache row j % ring_rows; 0: in row j
  int64_t T, start_pos;          // graph entry: T = the largest T, start_pos unused
  const int64_t* lens;           // graph entry: device {T, start_pos}; else null
  int64_t kv_capacity;           // rows per kv head in the cache
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

// Pair p -> kv head and token range; latest tokens (most keys) first.
__host__ __device__ inline Unit unit_of(int64_t T, int64_t start_pos, int Hkv, int tok_per_tile,
                                        int window, int units_per_head, int pidx) {
  Unit u;
  u.kh = pidx % Hkv;
  const int idx = units_per_head - 1 - pidx / Hkv;
  u.t0A = (int64_t)(2 * idx) * tok_per_tile;
  u.t0B = u.t0A + tok_per_tile;
  const int64_t t_end = (u.t0B + tok_per_tile < T) ? u.t0B + tok_per_tile : T;  // > t0A
  const int64_t pos_lo = start_pos + u.t0A;
  const int64_t pos_hi = start_pos + t_end - 1;
  int64_t kmin = 0;
  if (window > 0) kmin = (pos_lo - window + 1 > 0) ? pos_lo - window + 1 : 0;
  u.kt_first = kmin / kBN;
  u.n = (int)(pos_hi / kBN - u.kt_first + 1);
  return u;
}
__device__ __forceinline__ Unit unit_of(const Params& p, int pidx) {
  return unit_of(p.T, p.start_pos, p.Hkv, p.tok_per_tile, p.window, p.units_per_head, pidx);
}

// kShort (launches whose pairs hold few key tiles, where the set-up and the
// epilogue are a large part of each CTA): Q_B is loaded after the first K
// tile, so the first product waits for half of the query rows only, and the
// output is staged in the free Q buffer and written back in 512-byte runs.
// The long launches keep the plain order and direct stores, which measured
// ~1% faster there.
template <bool kFoldScale, bool kDyn, typename SchedT, bool kShort>
__global__ void __launch_bounds__(kThreads, 1)
bf16_d128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const Params p,
                 const __grid_constant__ SchedT sched) {
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
  const int cta = blockIdx.x;
  // Chunk length and position: kernel parameters, or (graph entry, kDyn) read
  // from device memory at run time, with the grid sized for the largest T.
  int64_t T = p.T, start_pos = p.start_pos;
  int units_per_head = p.units_per_head;
  if (kDyn) {
    T = p.lens[0];
    start_pos = p.lens[1];
    if (!lengths_ok(T, start_pos, p.T, p.kv_capacity, p.ring_rows, p.window)) {
      if (cta == 0 && threadIdx.x == 0) atomicOr(p.err, kErrLengths);
      return;
    }
    units_per_head = (int)(((T + p.tok_per_tile - 1) / p.tok_per_tile + 1) / 2);
    if (cta >= units_per_head * p.Hkv) return;  // the whole CTA: nothing set up yet
  }
  auto unit = [&](int pidx) -> Unit {
    return unit_of(T, start_pos, p.Hkv, p.tok_per_tile, p.window, units_per_head, pidx);
  };
  constexpr bool kHasTable = sizeof(SchedT) > sizeof(SchedLite);
  const bool table = kHasTable && (sched.mode == kTable);
  const int item_begin = table ? table_first(sched, cta) : 0;
  const int item_end = table ? table_first(sched, cta + 1) : 1;
  auto get_item = [&](int k) -> Item {
    if (table) return table_item(sched, k);
    Item it;
    if (sched.mode == kTail && cta >= sched.p1) {
      const int j = cta - sched.p1, r = j / sched.p2;
      it.pair = sched.p1 + j % sched.p2;
      const int n = unit(it.pair).n;
      it.kb = (int)((int64_t)n * r / sched.parts);
      it.ke = (int)((int64_t)n * (r + 1) / sched.parts);
      it.slot = j;
    } else {
      it.pair = cta;
      it.kb = 0;
      it.ke = unit(cta).n;
      it.slot = -1;
    }
    return it;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      // P and O-free: one arrival per softmax warp; all others: one arrival
      const bool per_warp = (i == kBarP || i == kBarP + 1 || i == kBarOFree || i == kBarOFree + 1);
      mbar_init(bar(i), per_warp ? 4u : 1u);
    }
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

  if (warp >= 8) {
   if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      // Each Q box is group x tok_per_tile rows of 128 bytes (zero-filled past T).
      const uint32_t q_bytes = 4u * 128u * (uint32_t)(p.group * p.tok_per_tile);
      uint32_t li = 0, nq = 0;
      bool ok = true, qb_pending = false;
      for (int k = item_begin; k < item_end && ok; ++k) {
        const Item it = get_item(k);
        const Unit u = unit(it.pair);
        if (nq > 0 && !(ok = mbar_wait(bar(kBarQFree), (nq - 1) & 1u, abort_flag, p.err, lim)))
          break;
        const int hq = u.kh * p.group;
        auto load_qb = [&](uint32_t b) {
          tma_load_3d(sbase + kSmemQ + kTileBytes, &tm_q, b, 0, hq, (int)u.t0B);
          tma_load_3d(sbase + kSmemQ + kTileBytes + kHalfBytes, &tm_q, b, 64, hq, (int)u.t0B);
        };
        mbar_arrive_expect_tx(bar(kBarQ), kShort ? q_bytes / 2 : q_bytes);
        tma_load_3d(sbase + kSmemQ, &tm_q, bar(kBarQ), 0, hq, (int)u.t0A);
        tma_load_3d(sbase + kSmemQ + kHalfBytes, &tm_q, bar(kBarQ), 64, hq, (int)u.t0A);
        if (!kShort) load_qb(bar(kBarQ));
        qb_pending = kShort;
        ++nq;
        for (int i = it.kb; i < it.ke && ok; ++i) {
          const int key0 = (int)((u.kt_first + i) * kBN);
          // A circular cache of a multiple of kBN rows never wraps inside a tile.
          const int row0 = p.ring_rows > 0 ? key0 % p.ring_rows : key0;
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t s = li % kSlots, ph = (li / kSlots) & 1u;
            if (!(ok = mbar_wait(bar(kBarEmpty + s), ph ^ 1u, abort_flag, p.err, lim))) break;
            const uint32_t dst = sbase + kSmemRing + s * kTileBytes;
            const CUtensorMap* map = kv ? &tm_v : &tm_k;
            mbar_arrive_expect_tx(bar(kBarFull + s), kTileBytes);
            tma_load_3d(dst, map, bar(kBarFull + s), 0, row0, u.kh);
            tma_load_3d(dst + kHalfBytes, map, bar(kBarFull + s), 64, row0, u.kh);
            ++li;
            if (kShort && qb_pending) {  // Q_B right after the item's first K tile
              qb_pending = false;
              mbar_arrive_expect_tx(bar(kBarQB), q_bytes / 2);
              load_qb(bar(kBarQB));
            }
          }
        }
      }
      // No copy may be in flight when the CTA exits.  On the normal path the
      // MMA thread has already consumed every load, so these return at once.
      if (nq > 0) mbar_wait(bar(kBarQ), (nq - 1) & 1u, abort_flag, p.err, lim, true);
      if (kShort && nq > 0 && !qb_pending)
        mbar_wait(bar(kBarQB), (nq - 1) & 1u, abort_flag, p.err, lim, true);
      const uint32_t first = li > (uint32_t)kSlots ? li - kSlots : 0;
      for (uint32_t j = first; j < li; ++j)
        mbar_wait(bar(kBarFull + j % kSlots), (j / kSlots) & 1u, abort_flag, p.err, lim, true);
    }
   } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (operands stay warp-uniform); one elected
    // lane issues each group of MMAs and each commit.
    {
      const uint32_t tSA = tmem + 0, tSB = tmem + 128, tOA = tmem + 256, tOB = tmem + 384;
      const uint64_t qdA = sdesc_sw128(sbase + kSmemQ, 16, 1024);
      const uint64_t qdB = sdesc_sw128(sbase + kSmemQ + kTileBytes, 16, 1024);
      uint32_t li = 0;  // ring index of the next K tile
      uint32_t gi = 0;  // key tiles done by this CTA (phase of the S and P barriers)
      uint32_t kk = 0;  // items done
      bool ok = true, issued = false;
      // O_X of the previous item must have been read by its epilogue before
      // the first P V product of the next item overwrites it.
      auto wait_o_free = [&](int X, int local_tile) -> bool {
        if (local_tile != 0 || kk == 0) return true;
        return mbar_wait_warp(bar(kBarOFree + X), (kk - 1) & 1u, abort_flag, p.err, lim);
      };
      for (int k = item_begin; k < item_end && ok; ++k) {
        const Item it = get_item(k);
        const int n = it.ke - it.kb;
        if (!(ok = mbar_wait_warp(bar(kBarQ), kk & 1u, abort_flag, p.err, lim))) break;
        tc_fence_after();
        for (int i = 0; i < n; ++i) {
          const uint32_t ks = li % kSlots;
          if (!(ok = mbar_wait_warp(bar(kBarFull + ks), (li / kSlots) & 1u, abort_flag, p.err, lim)))
            break;
          tc_fence_after();
          const uint32_t k_addr = sbase + kSmemRing + ks * kTileBytes;
          mma8_ss_kmajor<kHalfBytes / 16>(tSA, qdA, sdesc_sw128(k_addr, 16, 1024), kIdescQK, 0);
          issued = true;
          tc_commit_elect(bar(kBarS + 0));
          if (i > 0) {
            if (!(ok = mbar_wait_warp(bar(kBarP + 1), (gi - 1) & 1u, abort_flag, p.err, lim))) break;
            if (!(ok = wait_o_free(1, i - 1))) break;
            tc_fence_after();
            const uint32_t vs = (li - 1) % kSlots;  // V_{i-1}
            mma8_ts<2048 / 16>(tOB, tSB, sdesc_sw128(sbase + kSmemRing + vs * kTileBytes, kHalfBytes, 1024), kIdescPV,
                 (i - 1 > 0) ? 1u : 0u);
            tc_commit_elect(bar(kBarEmpty + vs));
          }
          if (kShort && i == 0) {
            if (!(ok = mbar_wait_warp(bar(kBarQB), kk & 1u, abort_flag, p.err, lim))) break;
            tc_fence_after();
          }
          mma8_ss_kmajor<kHalfBytes / 16>(tSB, qdB, sdesc_sw128(k_addr, 16, 1024), kIdescQK, 0);
          tc_commit_elect(bar(kBarS + 1));
          tc_commit_elect(bar(kBarEmpty + ks));
          if (i == n - 1) tc_commit_elect(bar(kBarQFree));
          const uint32_t vs = (li + 1) % kSlots;  // V_i
          if (!(ok = mbar_wait_warp(bar(kBarFull + vs), ((li + 1) / kSlots) & 1u, abort_flag, p.err,
                               lim)))
            break;
          if (!(ok = mbar_wait_warp(bar(kBarP + 0), gi & 1u, abort_flag, p.err, lim))) break;
          if (!(ok = wait_o_free(0, i))) break;
          tc_fence_after();
          mma8_ts<2048 / 16>(tOA, tSA, sdesc_sw128(sbase + kSmemRing + vs * kTileBytes, kHalfBytes, 1024), kIdescPV,
                 (i > 0) ? 1u : 0u);
          li += 2;
          ++gi;
        }
        if (!ok) break;
        // last product of tile B
        if (!(ok = mbar_wait_warp(bar(kBarP + 1), (gi - 1) & 1u, abort_flag, p.err, lim))) break;
        if (!(ok = wait_o_free(1, n - 1))) break;
        tc_fence_after();
        const uint32_t vs = (li - 1) % kSlots;
        mma8_ts<2048 / 16>(tOB, tSB, sdesc_sw128(sbase + kSmemRing + vs * kTileBytes, kHalfBytes, 1024), kIdescPV,
                 (n - 1 > 0) ? 1u : 0u);
        tc_commit_elect(bar(kBarEmpty + vs));
        tc_commit_elect(bar(kBarO + 0));
        tc_commit_elect(bar(kBarO + 1));
        ++kk;
      }
      if (issued) {
        // Everything issued must complete before TMEM is freed (this matters
        // when another role gave up early and skipped its wait on kBarO).
        tc_commit_elect(bar(kBarDrain));
        mbar_wait_warp(bar(kBarDrain), 0, abort_flag, p.err, lim, true);
      }
    }
   }
  } else {
    // ------------------------------------------------------------ softmax
    const int X = warp >> 2;        // 0: tile A, 1: tile B
    const int wq = warp & 3;        // lane quarter
    const int row = wq * 32 + lane;
    const int tok = row / p.group;
    const bool row_exists = tok < p.tok_per_tile;
    const int hrow = row % p.group;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)(X * 128);
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(X * 128);
    const float c = p.scale_log2;

    bool ok = true;
    if ((p.flags & kFlagForceTimeout) && X == 0) {
      // Test hook: wait on a barrier nothing signals, so the limit expires.
      ok = mbar_wait(bar(kBarDrain), 0, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    uint32_t gi = 0, kk = 0;
    for (int k = item_begin; k < item_end && ok; ++k, ++kk) {
      const Item it = get_item(k);
      const Unit u = unit(it.pair);
      const int n = it.ke - it.kb;
      // Positions and key indices fit in 32 bits (L < 2^31 - 4096).
      const int t0 = (int)(X ? u.t0B : u.t0A);
      const int pos_first = (int)start_pos + t0;
      // first key of this item's first tile, relative to the row's position
      int key_rel = (int)(u.kt_first + it.kb) * kBN - (pos_first + tok);

      float m_run = -INFINITY, l = 0.f;
      for (int i = 0; i < n; ++i, ++gi, key_rel += kBN) {
        ok = mbar_wait(bar(kBarS + X), gi & 1u, abort_flag, p.err, lim);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        tc_fence_after();

        uint32_t r0[32], r1[32], r2[32], r3[32];  // four loads in flight
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
        // Per-element mask unless the tile is visible to every row of the tile.
        const int key0_minus_first = key_rel + tok;  // key0 - pos_first
        const bool all_visible =
            (key0_minus_first + kBN - 1 <= 0) &&
            (p.window <= 0 || key0_minus_first > p.tok_per_tile - 1 - p.window);
        if (!all_visible) {
          const int hi = -key_rel;                                   // j - key0 <= pos - key0
          const int lo = p.window > 0 ? -key_rel - p.window : -1;    // j - key0 > lo
#pragma unroll
          for (int j = 0; j < 128; ++j)
            if (j > hi || j <= lo) x[j] = -INFINITY;
        }
        // Row max with three-input max instructions in 8 independent chains.
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

        // Raise the exponent base only when the new maximum exceeds it by > 2^8.
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_run + kRescaleThreshold) {
          alpha = ex2(m_run - mx);  // 0 while nothing was accumulated
          rescale = (i > 0) && (m_run != -INFINITY);
          m_run = mx;
        }
        const float base = (m_run == -INFINITY) ? 0.f : m_run;

        // P = 2^(s - base) as packed bf16 pairs; l gains the row sum of the
        // unrounded values (8 independent partial sums).
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
      if (!ok) break;

      ok = mbar_wait(bar(kBarO + X), kk & 1u, abort_flag, p.err, lim);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      const int64_t t = (int64_t)t0 + tok;
      const bool row_valid = row_exists && t < T;
      const int h = u.kh * p.group + hrow;
      if (kShort && !kHasTable && it.slot < 0) {
        // whole pair, the CTA's only item: this tile's Q buffer is free (every
        // S_X product has completed), so each warp stages its 32 output rows
        // there, 16-byte chunks rotated by row, and writes them back two rows
        // (512 contiguous bytes) per store instead of 32 scattered 16-byte pieces.
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint8_t* wbuf = smem + kSmemQ + X * kTileBytes + wq * (32 * 256);
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld(o);
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int chunk = (c0 >> 3) + j;
            *reinterpret_cast<uint4*>(wbuf + lane * 256 + ((chunk ^ (lane & 15)) << 4)) =
                make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          }
        }
        __syncwarp();
        const int ch = lane & 15;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const int rl = 2 * i + (lane >> 4);
          const uint4 val =
              *reinterpret_cast<const uint4*>(wbuf + rl * 256 + ((ch ^ (rl & 15)) << 4));
          const int r = wq * 32 + rl;
          const int tk = r / p.group;
          const int64_t tt = (int64_t)t0 + tk;
          if (tk < p.tok_per_tile && tt < T)
            *reinterpret_cast<uint4*>(p.out + tt * p.o_stride +
                                      (int64_t)(u.kh * p.group + r % p.group) * 128 + ch * 8) = val;
        }
      } else if (it.slot < 0) {
        // whole pair: normalise, round to bf16, store token-major
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow = p.out + (t * p.o_stride + h * (int64_t)128);
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
      } else {
        // part of a pair: unnormalised fp32 partial, its exponent base and sum.
        // Layout [column/4][row][4]: a warp's 32 rows store 512 contiguous bytes.
        float* slot = p.ws + (size_t)it.slot * kSlotFloats;
        const int R = X * kBM + row;
        float4* ocol = reinterpret_cast<float4*>(slot) + R;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            ocol[(size_t)(c0 / 4 + j) * kPairRows] =
                make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                            __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
        }
        slot[(size_t)kPairRows * 128 + R] = m_run;
        slot[(size_t)kPairRows * 128 + kPairRows + R] = l;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarOFree + X));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Combines the partial results of each split pair, in key order:
// m = max_i m_i, O = sum_i 2^(m_i - m) O_i, l = sum_i 2^(m_i - m) l_i, out = O / l.
// Block (e, g): merge entry e, columns 16 g .. 16 g + 15; thread R owns row R
// (the partials' [column/4][row][4] layout makes every load coalesced across
// the rows of a warp).  Up to kMergeUnroll pieces' loads are in flight at once.
constexpr int kMergeCols = 16;
constexpr int kMergeUnroll = 4;

template <typename MS>
__global__ void __launch_bounds__(kPairRows)
merge_kernel(const Params p, const __grid_constant__ MS ms) {
  MergeEntry e;
  if (ms.tail) {
    e.pair = ms.p1 + (int)blockIdx.x;
    e.first = 0;
    e.count = ms.parts;
  } else {
    e = merge_entry(ms, (int)blockIdx.x);
  }
  auto slot_of = [&](int i) -> int {
    return ms.tail ? i * ms.p2 + (int)blockIdx.x : merge_slot(ms, e.first + i);
  };
  const Unit u = unit_of(p, e.pair);
  const int R = threadIdx.x;
  const int X = R / kBM, row = R % kBM;
  const int tok = row / p.group;
  const int64_t t = (X ? u.t0B : u.t0A) + tok;
  if (tok >= p.tok_per_tile || t >= p.T) return;
  const int h = u.kh * p.group + row % p.group;
  const int cq0 = blockIdx.y * (kMergeCols / 4);   // first column quad
  const size_t off_m = (size_t)kPairRows * 128 + R, off_l = off_m + kPairRows;

  float m = -INFINITY;
  for (int i0 = 0; i0 < e.count; i0 += kMergeUnroll) {
    float mi[kMergeUnroll];
#pragma unroll
    for (int j = 0; j < kMergeUnroll; ++j)
      mi[j] = (i0 + j < e.count)
                  ? p.ws[(size_t)slot_of(i0 + j) * kSlotFloats + off_m]
                  : -INFINITY;
#pragma unroll
    for (int j = 0; j < kMergeUnroll; ++j) m = fmaxf(m, mi[j]);
  }
  const float mb = (m == -INFINITY) ? 0.f : m;
  float4 acc[kMergeCols / 4];
#pragma unroll
  for (int q = 0; q < kMergeCols / 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  for (int i0 = 0; i0 < e.count; i0 += kMergeUnroll) {
#pragma unroll
    for (int j = 0; j < kMergeUnroll; ++j) {
      if (i0 + j >= e.count) break;
      const float* slot = p.ws + (size_t)slot_of(i0 + j) * kSlotFloats;
      const float w = ex2(slot[off_m] - mb);  // 0 for a piece that saw no visible key
      l = fmaf(w, slot[off_l], l);
      const float4* ocol = reinterpret_cast<const float4*>(slot) + R;
#pragma unroll
      for (int q = 0; q < kMergeCols / 4; ++q) {
        const float4 o = ocol[(size_t)(cq0 + q) * kPairRows];
        acc[q].x = fmaf(w, o.x, acc[q].x);
        acc[q].y = fmaf(w, o.y, acc[q].y);
        acc[q].z = fmaf(w, o.z, acc[q].z);
        acc[q].w = fmaf(w, o.w, acc[q].w);
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint32_t wv[kMergeCols / 2];
#pragma unroll
  for (int q = 0; q < kMergeCols / 4; ++q) {
    wv[2 * q] = pack_bf16x2(acc[q].x * inv, acc[q].y * inv);
    wv[2 * q + 1] = pack_bf16x2(acc[q].z * inv, acc[q].w * inv);
  }
  uint4* dst = reinterpret_cast<uint4*>(p.out + t * p.o_stride + h * (int64_t)128 + cq0 * 4);
#pragma unroll
  for (int q = 0; q < kMergeCols / 8; ++q)
    dst[q] = make_uint4(wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
}

// ------------------------------------------------------------------ host
struct Plan {
  bool balanced = false;
  int grid = 0;
  size_t ws_bytes = 0;
  Sched sched;
  MergeSched merge;
};

struct Shape {
  int64_t T, start_pos;
  int H, Hkv, group, tok_per_tile, window, units_per_head, pairs;
};

bool make_shape(const Call& c, Shape* s) {
  s->T = c.T;
  s->start_pos = c.start_pos;
  s->H = c.H;
  s->Hkv = c.Hkv;
  s->group = c.H / c.Hkv;
  s->tok_per_tile = kBM / s->group;  // group <= 128 checked by the caller
  s->window = c.window;
  const int64_t tiles = (c.T + s->tok_per_tile - 1) / s->tok_per_tile;
  const int64_t units = (tiles + 1) / 2;
  const int64_t L = c.start_pos + c.T;
  if (units * c.Hkv > 0x7fffffff || L + kBN > 0x7fffffff ||
      c.T + 2 * (int64_t)s->tok_per_tile > 0x7fffffff)
    return false;
  s->units_per_head = (int)units;
  s->pairs = (int)(units * c.Hkv);
  return true;
}

// Balanced schedule.  Each item costs its key tiles plus a fixed overhead
// (reloading Q, refilling the pipeline, the epilogue), in key-tile units.
// The pairs, in order, are cut into at most `ctas` consecutive runs of items
// whose costs do not exceed a common budget; the smallest budget that covers
// all pairs is found by bisection.  Returns false if the tables would
// overflow (the caller then uses the plain schedule).
constexpr int kItemOverheadTiles = 3;

// Greedy cut for a given budget; returns the number of CTAs used (or
// ctas + 1 if the budget is too small).  With `plan` it also fills the tables.
int cut(const std::vector<int>& n, int64_t budget, int ctas, Plan* plan, int* n_items,
        int* n_slots, std::vector<std::vector<int>>* pieces) {
  const int pairs = (int)n.size();
  int c = 0, items = 0, slots = 0;
  int q = 0, done = 0;  // pair q, tiles of it already assigned
  while (q < pairs) {
    if (c >= ctas) return ctas + 1;
    int64_t left = budget;
    if (plan) plan->sched.cta_first[c] = items;
    while (q < pairs && left > kItemOverheadTiles) {
      const int rest = n[q] - done;
      const int take = (int)std::min<int64_t>(rest, left - kItemOverheadTiles);
      if (plan) {
        if (items >= kMaxItems) return ctas + 1;
        Item& it = plan->sched.items[items];
        it.pair = q;
        it.kb = done;
        it.ke = done + take;
        const bool whole = (done == 0 && take == n[q]);
        it.slot = whole ? -1 : slots;
        if (!whole) (*pieces)[q].push_back(slots);
      }
      ++items;
      if (!(done == 0 && take == n[q])) ++slots;
      left -= take + kItemOverheadTiles;
      done += take;
      if (done == n[q]) {
        ++q;
        done = 0;
      }
    }
    ++c;
  }
  if (plan) plan->sched.cta_first[c] = items;
  *n_items = items;
  *n_slots = slots;
  return c;
}

bool plan_balanced(const Shape& s, int ctas, Plan* plan) {
  if (s.pairs <= 0) return false;
  if (ctas > kMaxCtas) ctas = kMaxCtas;
  std::vector<int> n(s.pairs);
  int64_t W = 0;
  int nmax = 0;
  for (int pi = 0; pi < s.pairs; ++pi) {
    n[pi] = unit_of(s.T, s.start_pos, s.Hkv, s.tok_per_tile, s.window, s.units_per_head, pi).n;
    W += n[pi];
    nmax = std::max(nmax, n[pi]);
  }
  // smallest budget (>= one tile plus overhead) that fits in `ctas` CTAs
  int64_t lo = kItemOverheadTiles + 1, hi = W + (int64_t)s.pairs * kItemOverheadTiles + 1;
  int items = 0, slots = 0;
  while (lo < hi) {
    const int64_t mid = (lo + hi) / 2;
    if (cut(n, mid, ctas, nullptr, &items, &slots, nullptr) <= ctas)
      hi = mid;
    else
      lo = mid + 1;
  }
  std::vector<std::vector<int>> pieces(s.pairs);
  const int used = cut(n, lo, ctas, plan, &items, &slots, &pieces);
  if (used > ctas || items > kMaxItems || slots > kMaxPieces) return false;
  MergeSched& ms = plan->merge;
  int ne = 0, np = 0;
  for (int q = 0; q < s.pairs; ++q) {
    if (pieces[q].empty()) continue;
    if (ne >= kMaxMerge) return false;
    MergeEntry& e = ms.e[ne++];
    e.pair = q;
    e.first = np;
    e.count = (int)pieces[q].size();
    e.pad = 0;
    for (int sl : pieces[q]) ms.slots[np++] = sl;
  }
  ms.num = ne;
  ms.tail = 0;
  plan->sched.mode = kTable;
  plan->balanced = true;
  plan->grid = used;
  plan->ws_bytes = (size_t)slots * kSlotBytes;
  return true;
}

// Cost of the merge kernel and of writing and reading the partials, in
// key-tile units (a measured few microseconds).
constexpr int64_t kMergeCostTiles = 3;

// Makespan, in key-tile units, of CTAs with the given costs launched in order:
// the hardware starts each on the first SM that frees up.
int64_t list_makespan(const std::vector<int64_t>& costs, int sms) {
  std::vector<int64_t> free_at((size_t)std::max(sms, 1), 0);  // min-heap of SM finish times
  int64_t makespan = 0;
  for (int64_t cost : costs) {
    std::pop_heap(free_at.begin(), free_at.end(), std::greater<int64_t>());
    free_at.back() += cost;
    makespan = std::max(makespan, free_at.back());
    std::push_heap(free_at.begin(), free_at.end(), std::greater<int64_t>());
  }
  return makespan;
}

std::vector<int> pair_tiles(const Shape& s) {
  std::vector<int> n(s.pairs);
  for (int pi = 0; pi < s.pairs; ++pi)
    n[pi] = unit_of(s.T, s.start_pos, s.Hkv, s.tok_per_tile, s.window, s.units_per_head, pi).n;
  return n;
}

// Plain schedule: one CTA per pair.
int64_t plain_makespan(const std::vector<int>& n, int sms) {
  std::vector<int64_t> costs(n.size());
  for (size_t i = 0; i < n.size(); ++i) costs[i] = n[i] + kItemOverheadTiles;
  return list_makespan(costs, sms);
}

// Whether the balanced schedule may be used.  Its CTAs do not walk a kv
// head's keys in step, so when many pairs of a large cache are in flight
// each CTA would stream its keys from DRAM; it is allowed when the K/V cache
// stays in L2, or when there are no more pairs than SMs (then each CTA reads
// its own key range once).
constexpr int64_t kBalancedKvBytesMax = 96ll << 20;

bool balanced_allowed(const Shape& s, int sms) {
  const int64_t kv_bytes = 2ll * s.Hkv * (s.start_pos + s.T) * 128 * 2;
  return kv_bytes <= kBalancedKvBytesMax || s.pairs <= sms;
}

// Tail-split schedule for more pairs than SMs: the whole waves of pairs run
// whole (their CTAs move through the keys together, as in the plain
// schedule); each pair of the last, partial wave is cut into `parts` equal
// key ranges run as separate CTAs, part by part, so that the CTAs of one part
// again read the same keys at about the same time.  Returns false if no cut
// applies.
constexpr int kMaxTailParts = 8;

bool plan_tail(const Shape& s, const std::vector<int>& n, int sms, Plan* plan,
               int64_t* makespan) {
  if (s.pairs <= sms) return false;
  const int p1 = sms * (s.pairs / sms), p2 = s.pairs - p1;
  if (p2 == 0 || p2 > kMaxMerge) return false;
  int nmin = n[p1];
  for (int q = p1; q < s.pairs; ++q) nmin = std::min(nmin, n[q]);
  int best_parts = 0;
  int64_t best = INT64_MAX;
  for (int parts = 2; parts <= kMaxTailParts && parts <= nmin; ++parts) {
    std::vector<int64_t> costs;
    costs.reserve(p1 + (size_t)p2 * parts);
    for (int q = 0; q < p1; ++q) costs.push_back(n[q] + kItemOverheadTiles);
    for (int r = 0; r < parts; ++r)
      for (int e = 0; e < p2; ++e) {
        const int64_t nq = n[p1 + e];
        costs.push_back(nq * (r + 1) / parts - nq * r / parts + kItemOverheadTiles);
      }
    const int64_t m = list_makespan(costs, sms) + kMergeCostTiles;
    if (m < best) {
      best = m;
      best_parts = parts;
    }
  }
  if (best_parts == 0) return false;
  plan->sched.mode = kTail;
  plan->sched.p1 = p1;
  plan->sched.p2 = p2;
  plan->sched.parts = best_parts;
  plan->merge.tail = 1;
  plan->merge.num = p2;
  plan->merge.p1 = p1;
  plan->merge.p2 = p2;
  plan->merge.parts = best_parts;
  plan->balanced = true;
  plan->grid = p1 + p2 * best_parts;
  plan->ws_bytes = (size_t)p2 * best_parts * kSlotBytes;
  *makespan = best;
  return true;
}

// Split of every pair, for no more pairs than SMs: each pair is cut into
// `parts` equal key ranges run part by part (CTA r * pairs + e runs part r of
// pair e: the tail-split layout with no whole pairs), in one wave.  The CTAs
// of one part start together, so the pairs of a kv head read each key range
// at about the same time and L2 serves the second read; the balanced
// table's runs, cut at a running budget, read the same keys at different
// times (measured: twice the algorithmic K/V bytes from DRAM on a 128-token
// chunk at 63k).
constexpr int kMaxSplitParts = 64;

bool plan_split_all(const Shape& s, const std::vector<int>& n, int sms, Plan* plan,
                    int64_t* makespan) {
  if (s.pairs <= 0 || s.pairs > sms || s.pairs > kMaxMerge) return false;
  int nmin = n[0];
  for (int v : n) nmin = std::min(nmin, v);
  const int pmax = std::min(std::min(kMaxSplitParts, nmin), sms / s.pairs);
  int best_parts = 0;
  int64_t best = INT64_MAX;
  for (int parts = 2; parts <= pmax; ++parts) {
    std::vector<int64_t> costs;
    costs.reserve((size_t)s.pairs * parts);
    for (int r = 0; r < parts; ++r)
      for (int e = 0; e < s.pairs; ++e) {
        const int64_t nq = n[e];
        costs.push_back(nq * (r + 1) / parts - nq * r / parts + kItemOverheadTiles);
      }
    const int64_t m = list_makespan(costs, sms) + kMergeCostTiles;
    if (m < best) {
      best = m;
      best_parts = parts;
    }
  }
  if (best_parts == 0) return false;
  plan->sched.mode = kTail;
  plan->sched.p1 = 0;
  plan->sched.p2 = s.pairs;
  plan->sched.parts = best_parts;
  plan->merge.tail = 1;
  plan->merge.num = s.pairs;
  plan->merge.p1 = 0;
  plan->merge.p2 = s.pairs;
  plan->merge.parts = best_parts;
  plan->balanced = true;
  plan->grid = s.pairs * best_parts;
  plan->ws_bytes = (size_t)s.pairs * best_parts * kSlotBytes;
  *makespan = best;
  return true;
}

// Picks the schedule with the smallest estimated makespan.  A workspace
// schedule must beat the plain one by a margin: 5% for the tail split (its
// CTAs still read the keys in step; measured ~11% faster on 64k and 128k
// chunks, where the estimate is 14%) and 15% for the balanced table (whose
// CTAs read unrelated key ranges).  Returns true (and fills *plan) for a
// workspace schedule, false for plain.
bool choose_schedule(const Shape& s, int sms, Plan* plan) {
  const std::vector<int> n = pair_tiles(s);
  const int64_t plain = plain_makespan(n, sms);
  int64_t best = INT64_MAX;  // estimated makespan of the chosen workspace schedule
  bool chosen = false;
  {
    std::unique_ptr<Plan> t(new Plan());
    int64_t m = 0;
    if (plan_tail(s, n, sms, t.get(), &m) && m < plain * 95 / 100) {
      *plan = *t;
      best = m;
      chosen = true;
    }
  }
  if (balanced_allowed(s, sms)) {
    std::unique_ptr<Plan> b(new Plan());
    if (plan_balanced(s, sms, b.get()) && b->merge.num > 0) {
      int64_t budget = 0;
      for (int c = 0; c < b->grid; ++c) {
        int64_t cost = 0;
        for (int k = b->sched.cta_first[c]; k < b->sched.cta_first[c + 1]; ++k)
          cost += b->sched.items[k].ke - b->sched.items[k].kb + kItemOverheadTiles;
        budget = std::max(budget, cost);
      }
      const int64_t m = budget + kMergeCostTiles;
      if (m < plain * 85 / 100 && m < best) {
        *plan = *b;
        best = m;
        chosen = true;
      }
    }
  }
  {
    // preferred to the balanced table unless its estimate is over 15% longer
    // (the estimate does not see the balanced table's second DRAM read); any
    // other choice it must beat outright
    std::unique_ptr<Plan> a(new Plan());
    int64_t m = 0;
    const bool over_table = chosen && plan->sched.mode == kTable;
    if (plan_split_all(s, n, sms, a.get(), &m) && m < plain * 85 / 100 &&
        (!chosen || (over_table ? m * 100 <= best * 115 : m < best))) {
      *plan = *a;
      best = m;
      chosen = true;
    }
  }
  return chosen;
}

}  // namespace

// Workspace schedules, cached per shape: planning simulates the SMs (tens of
// microseconds for long chunks), and callers repeat shapes layer after layer.
// A null entry means the plain schedule.  Most recently used first.
struct PlanKey {
  int64_t T, start_pos;
  int H, Hkv, window, sms;
  bool operator==(const PlanKey& o) const {
    return T == o.T && start_pos == o.start_pos && H == o.H && Hkv == o.Hkv &&
           window == o.window && sms == o.sms;
  }
};
constexpr size_t kPlanCacheEntries = 32;
std::mutex g_plan_mutex;
std::vector<std::pair<PlanKey, std::shared_ptr<const Plan>>> g_plans;

std::shared_ptr<const Plan> workspace_plan(const Shape& s, int sms) {
  const PlanKey key{s.T, s.start_pos, s.H, s.Hkv, s.window, sms};
  {
    std::lock_guard<std::mutex> lk(g_plan_mutex);
    for (size_t i = 0; i < g_plans.size(); ++i)
      if (g_plans[i].first == key) {
        std::shared_ptr<const Plan> hit = g_plans[i].second;
        std::rotate(g_plans.begin(), g_plans.begin() + i, g_plans.begin() + i + 1);
        return hit;
      }
  }
  std::shared_ptr<Plan> plan = std::make_shared<Plan>();
  std::shared_ptr<const Plan> made;
  if (choose_schedule(s, sms, plan.get())) made = plan;
  std::lock_guard<std::mutex> lk(g_plan_mutex);
  g_plans.insert(g_plans.begin(), {key, made});
  if (g_plans.size() > kPlanCacheEntries) g_plans.pop_back();
  return made;
}

// Host replay of the kernel's work assignment for one shape and SM count,
// with the invariants every schedule must keep (see pfa_debug_check_schedule
// in include/pfa.h).  Returns 0, or the number of the first failed check.
int check_schedule_bf16_d128(const Call& c, int sms, int* schedule, int* ctas) {
  Shape s;
  if (!make_shape(c, &s)) return 1;
  std::unique_ptr<Plan> plan(new Plan());
  if (!choose_schedule(s, sms, plan.get())) {
    plan->balanced = false;
    plan->sched.mode = kPlain;
    plan->grid = s.pairs;
    plan->ws_bytes = 0;
  }
  const Sched& sc = plan->sched;
  *schedule = sc.mode == kTail ? 2 : (sc.mode == kTable ? 1 : 0);
  *ctas = plan->grid;
  const std::vector<int> n = pair_tiles(s);
  const int64_t L = s.start_pos + s.T;
  // items of every CTA, as the kernel derives them
  struct Got { int pair, kb, ke, slot; };
  std::vector<Got> all;
  for (int cta = 0; cta < plan->grid; ++cta) {
    if (sc.mode == kTable) {
      if (cta >= kMaxCtas || sc.cta_first[cta] > sc.cta_first[cta + 1] ||
          sc.cta_first[cta + 1] > kMaxItems)
        return 2;
      for (int k = sc.cta_first[cta]; k < sc.cta_first[cta + 1]; ++k)
        all.push_back({sc.items[k].pair, sc.items[k].kb, sc.items[k].ke, sc.items[k].slot});
    } else if (sc.mode == kTail && cta >= sc.p1) {
      const int j = cta - sc.p1, r = j / sc.p2, pair = sc.p1 + j % sc.p2;
      if (pair >= s.pairs) return 3;
      all.push_back({pair, (int)((int64_t)n[pair] * r / sc.parts),
                     (int)((int64_t)n[pair] * (r + 1) / sc.parts), j});
    } else {
      if (cta >= s.pairs) return 3;
      all.push_back({cta, 0, n[cta], -1});
    }
  }
  // every key tile of every pair exactly once; whole-pair items direct,
  // partial items in distinct slots that fit the workspace
  std::vector<std::vector<std::pair<int, int>>> ranges(s.pairs);
  std::vector<int> slot_used(kMaxPieces * 16, 0);
  const size_t nslots = plan->ws_bytes / kSlotBytes;
  for (const Got& g : all) {
    if (g.pair < 0 || g.pair >= s.pairs || g.kb < 0 || g.ke > n[g.pair] || g.kb >= g.ke) return 4;
    const bool whole = g.kb == 0 && g.ke == n[g.pair];
    if (g.slot < 0 && !whole) return 5;
    if (g.slot >= 0) {
      if ((size_t)g.slot >= nslots || (size_t)g.slot >= slot_used.size() || slot_used[g.slot]++)
        return 6;
    }
    ranges[g.pair].emplace_back(g.kb, g.ke);
  }
  for (int q = 0; q < s.pairs; ++q) {
    std::sort(ranges[q].begin(), ranges[q].end());
    int at = 0;
    for (const auto& r : ranges[q]) {
      if (r.first != at) return 7;
      at = r.second;
    }
    if (at != n[q]) return 7;
    // key coordinates of the pair's tiles stay inside the cache, and each
    // tile holds a key some row of the pair sees
    const Unit u = unit_of(s.T, s.start_pos, s.Hkv, s.tok_per_tile, s.window, s.units_per_head, q);
    if (u.t0A < 0 || u.t0A >= s.T) return 8;
    const int64_t pos_lo = s.start_pos + u.t0A;
    const int64_t kmin = s.window > 0 ? std::max<int64_t>(0, pos_lo - s.window + 1) : 0;
    for (int i = 0; i < n[q]; ++i) {
      const int64_t key0 = (u.kt_first + i) * kBN;
      if (key0 < 0 || key0 >= L || key0 + kBN - 1 < kmin) return 9;
    }
  }
  // the merge kernel sees every split pair once, with its pieces in key order
  if (plan->balanced) {
    const MergeSched& ms = plan->merge;
    std::vector<int> merged(s.pairs, 0);
    for (int e = 0; e < ms.num; ++e) {
      int pair, count;
      std::vector<int> slots;
      if (ms.tail) {
        pair = ms.p1 + e;
        count = ms.parts;
        for (int r = 0; r < count; ++r) slots.push_back(r * ms.p2 + e);
      } else {
        pair = ms.e[e].pair;
        count = ms.e[e].count;
        for (int r = 0; r < count; ++r) slots.push_back(ms.slots[ms.e[e].first + r]);
      }
      if (pair < 0 || pair >= s.pairs || merged[pair]++) return 10;
      std::vector<std::pair<int, int>> pieces;  // (kb, slot) of the pair's partial items
      for (const Got& g : all)
        if (g.pair == pair && g.slot >= 0) pieces.emplace_back(g.kb, g.slot);
      std::sort(pieces.begin(), pieces.end());
      if ((int)pieces.size() != count) return 11;
      for (int r = 0; r < count; ++r)
        if (pieces[r].second != slots[r]) return 11;
    }
    for (int q = 0; q < s.pairs; ++q)
      if ((ranges[q].size() > 1) != (merged[q] > 0)) return 12;
  } else {
    for (const Got& g : all)
      if (g.slot >= 0) return 12;
  }
  return 0;
}

size_t workspace_bytes_bf16_d128(const Call& c, int* schedule) {
  if (schedule) *schedule = 0;
  Shape s;
  if (!make_shape(c, &s)) return 0;
  const std::shared_ptr<const Plan> plan = workspace_plan(s, c.num_sms);
  if (!plan) return 0;
  if (schedule) *schedule = plan->sched.mode == kTail ? 2 : 1;
  return plan->ws_bytes;
}

// One-time per-device set-up of a kernel variant: the shared-memory opt-in.
int setup_kernel(const void* fn) {
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) !=
      cudaSuccess)
    return kErrLaunch;
  return kOk;
}

int launch_bf16_d128(const Call& c) {
  static DeviceOnce setup;
  const int sr = setup.run(c.device, [] {
    const void* fns[] = {
        (const void*)bf16_d128_kernel<true, false, SchedLite, false>,
        (const void*)bf16_d128_kernel<false, false, SchedLite, false>,
        (const void*)bf16_d128_kernel<true, false, SchedLite, true>,
        (const void*)bf16_d128_kernel<false, false, SchedLite, true>,
        (const void*)bf16_d128_kernel<true, false, Sched, false>,
        (const void*)bf16_d128_kernel<false, false, Sched, false>,
        (const void*)bf16_d128_kernel<true, true, SchedLite, false>,
        (const void*)bf16_d128_kernel<false, true, SchedLite, false>};
    for (const void* fn : fns)
      if (setup_kernel(fn) != kOk) return kErrLaunch;
    return kOk;
  });
  if (sr != kOk) return sr;
  Shape s;
  if (!make_shape(c, &s)) return kErrShape;

  // A workspace schedule when the caller gave a large enough workspace, else
  // the plain one.
  std::shared_ptr<const Plan> wplan;
  if (c.ws != nullptr && c.lens == nullptr) {
    wplan = workspace_plan(s, c.num_sms);
    if (wplan && wplan->ws_bytes > c.ws_bytes) wplan.reset();
  }
  const int grid_ctas = wplan ? wplan->grid : s.pairs;
  const bool table = wplan && wplan->sched.mode == kTable;
  SchedLite lite{kPlain, 0, 0, 0};
  if (wplan) lite = SchedLite{wplan->sched.mode, wplan->sched.p1, wplan->sched.p2, wplan->sched.parts};

  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {128, (uint64_t)c.H, (uint64_t)c.T};
    const uint64_t strides[2] = {128 * 2, (uint64_t)c.qkv_dim * 2};
    const uint32_t box[3] = {64, (uint32_t)s.group, (uint32_t)s.tok_per_tile};
    if (encode_tmap_bf16_3d(&tq, c.q, dims, strides, box)) return kErrLaunch;
  }
  {
    // Rows past the written part of the cache read as zeros.
    const uint64_t dims[3] = {128, (uint64_t)cache_rows_written(c), (uint64_t)c.Hkv};
    const uint64_t strides[2] = {128 * 2, (uint64_t)c.max_seq_len * 128 * 2};
    const uint32_t box[3] = {64, (uint32_t)kBN, 1};
    if (encode_tmap_bf16_3d(&tk, c.k, dims, strides, box)) return kErrLaunch;
    if (encode_tmap_bf16_3d(&tv, c.v, dims, strides, box)) return kErrLaunch;
  }
  Params p;
  p.out = static_cast<__nv_bfloat16*>(c.out);
  p.ws = static_cast<float*>(c.ws);
  p.o_stride = c.qkv_dim;
  p.ring_rows = ring_rows(c);
  p.T = c.T;
  p.start_pos = c.start_pos;
  p.lens = c.lens;
  p.kv_capacity = c.max_seq_len;
  p.H = c.H;
  p.Hkv = c.Hkv;
  p.group = s.group;
  p.tok_per_tile = s.tok_per_tile;
  p.window = c.window;
  p.units_per_head = s.units_per_head;
  p.scale_log2 = (float)((double)c.scale * 1.4426950408889634);
  p.err = c.err;
  p.wait_limit_ns = c.wait_limit_ns;
  p.flags = c.flags;
  const dim3 grid((unsigned)grid_ctas);
  const bool fold = p.scale_log2 > 0.f;
  // Short launches: plain schedule and at most kShortTiles key tiles per pair.
  const bool short_launch = !wplan && unit_of(s.T, s.start_pos, s.Hkv, s.tok_per_tile, s.window,
                                              s.units_per_head, 0).n <= kShortTiles;
  if (c.lens) {
    if (fold)
      bf16_d128_kernel<true, true, SchedLite, false>
          <<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p, lite);
    else
      bf16_d128_kernel<false, true, SchedLite, false>
          <<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p, lite);
  } else if (table) {
    if (fold)
      bf16_d128_kernel<true, false, Sched, false>
          <<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p, wplan->sched);
    else
      bf16_d128_kernel<false, false, Sched, false>
          <<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p, wplan->sched);
  } else if (short_launch) {
    if (fold)
      bf16_d128_kernel<true, false, SchedLite, true>
          <<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p, lite);
    else
      bf16_d128_kernel<false, false, SchedLite, true>
          <<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p, lite);
  } else if (fold) {
    bf16_d128_kernel<true, false, SchedLite, false>
        <<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p, lite);
  } else {
    bf16_d128_kernel<false, false, SchedLite, false>
        <<<grid, kThreads, kSmemAlloc, c.stream>>>(tq, tk, tv, p, lite);
  }
  if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
  if (wplan && wplan->balanced && wplan->merge.num > 0) {
    const MergeSched& ms = wplan->merge;
    const dim3 mgrid((unsigned)ms.num, 128 / kMergeCols);
    if (ms.tail)
      merge_kernel<MergeLite><<<mgrid, kPairRows, 0, c.stream>>>(
          p, MergeLite{ms.num, ms.tail, ms.p1, ms.p2, ms.parts});
    else
      merge_kernel<MergeSched><<<mgrid, kPairRows, 0, c.stream>>>(p, ms);
    if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
  }
  return kOk;
}

}  // namespace pfa
