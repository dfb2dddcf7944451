// pfa_tf32_d128.cu -- fp32 prefill attention, head_dim 128, on the sm_103a
// tensor cores with the three-product TF32 split ("3xTF32").
//
// Operation (gnosis "Prefill attention -> GPU: handoff", section "GPU design",
// steps 1-3, fused; accuracy bar max |gpu - cpu| <= 1e-4 of its section
// "Implementation status"): per query row, scores against the visible keys of
// its kv head, scale, causal (+ window) mask, softmax, weighted sum of V.
//
// A tf32 operand keeps 10 mantissa bits, too few for the 1e-4 bar.  Every
// fp32 operand x is therefore split into hi = x with the low 13 mantissa bits
// cleared (exactly a tf32 value) and lo = x - hi (exact in fp32), and each
// product is formed as  hi*hi + hi*lo + lo*hi  with fp32 accumulation; the
// dropped lo*lo term and the tf32 rounding of lo are ~2^-20 relative.
//
// CTA = one kv head x one 128-row query tile (all `group` heads of the kv
// head for 128/group consecutive tokens; row r -> token r/group, head
// r%group), latest tokens first.  Key tiles of 64.
//
// Warp roles (9 warps):
//   warps 0-3  rows of the tile (TMEM lanes 0-127, one row per thread): split
//              Q into tensor memory once, then the online softmax of every key
//              tile, then the epilogue
//   warps 4-7  converters: read K and V tiles from global memory, split them
//              into hi/lo and write the tensor-core operand layouts (K as is,
//              V transposed so that its contraction index, the key, is the
//              contiguous one) into a 3-slot shared-memory ring
//   warp  8    TMEM allocator and MMA issuer (converged warp, elected lane)
//
// Tensor memory (512 columns, fp32 cells):
//   [  0,128) Q_hi   [128,256) Q_lo        (A operand of S = Q K^T)
//   [256,320) S, then P_hi                  (A operand of O += P V)
//   [320,384) P_lo
//   [384,512) O
// Issue order per key tile i: S(i) = Q_hi K_hi + Q_hi K_lo + Q_lo K_hi, then
// O += P_hi V_hi + P_hi V_lo + P_lo V_hi.  S(i+1) overwrites P_hi(i) only after
// O += P(i) V was issued (the tensor core executes in issue order), and the
// commit that signals S(i) covers P(i-1) V, so the softmax may rescale O.
//
// Online softmax in the log2 domain with the lazy rescale of the bf16
// kernels (the exponent base rises only when a row maximum exceeds it by more
// than 2^8); masks come from indices; every wait is bounded.
#include "pfa_internal.h"
#include "pfa_ptx.cuh"

#include <cmath>

namespace pfa {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                  // query rows per CTA
constexpr int kBN = 64;                   // keys per tile
constexpr int kThreads = 288;
constexpr int kOpSlots = 3;               // operand ring depth (tiles)
constexpr int kPartBytes = 32768;         // one hi or lo operand tile (fp32)
constexpr int kSlotBytes = 2 * kPartBytes;
constexpr int kSmemBars = kOpSlots * kSlotBytes;  // 196608
constexpr int kSmemAlloc = kSmemBars + 256 + 1024;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// barriers
constexpr int kBarQ = 0;                      // Q split into TMEM (4 warp arrivals)
constexpr int kBarFull = 1;                   // kOpSlots: operand tile written (4 arrivals)
constexpr int kBarEmpty = kBarFull + kOpSlots;  // kOpSlots: operand tile consumed (commit)
constexpr int kBarS = kBarEmpty + kOpSlots;   // S(i) complete (commit)
constexpr int kBarP = kBarS + 1;              // P(i) in TMEM (4 arrivals)
constexpr int kBarO = kBarP + 1;              // all products complete (commit)
constexpr int kBarDrain = kBarO + 1;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kOffTmemSlot = kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
static_assert(kOffAbort + 4 <= 256, "barrier area");

constexpr uint32_t kColQHi = 0, kColQLo = 128, kColS = 256, kColPLo = 320, kColO = 384;
constexpr uint32_t kIdescQK = idesc_tf32_f32(kBM, kBN);
constexpr uint32_t kIdescPV = idesc_tf32_f32(kBM, kD);

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

__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

__global__ void __launch_bounds__(kThreads, 1) tf32_d128_kernel(const Params p) {
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

  // work unit: (kv head, query tile); latest tokens first
  const int kh = (int)blockIdx.x % p.Hkv;
  const int tile = tiles_per_head - 1 - (int)blockIdx.x / p.Hkv;
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
      const bool per_warp = (i == kBarQ || i == kBarP || (i >= kBarFull && i < kBarFull + kOpSlots));
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

  if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = mbar_wait_warp(bar(kBarQ), 0, abort_flag, p.err, lim);
    bool issued = false;
    tc_fence_after();
    uint32_t li = 0;  // operand tiles consumed
    const uint32_t tS = tmem + kColS, tO = tmem + kColO;
    for (int i = 0; i < n && ok; ++i) {
      // S = Q_hi K_hi + Q_hi K_lo + Q_lo K_hi
      {
        const uint32_t s = li % kOpSlots;
        if (!(ok = mbar_wait_warp(bar(kBarFull + s), (li / kOpSlots) & 1u, abort_flag, p.err, lim)))
          break;
        tc_fence_after();
        const uint32_t hi = sbase + s * kSlotBytes, lo = hi + kPartBytes;
        const uint32_t qa[3] = {tmem + kColQHi, tmem + kColQHi, tmem + kColQLo};
        const uint32_t kb[3] = {hi, lo, hi};
#pragma unroll
        for (int prod = 0; prod < 3; ++prod) {
          // four 32-column spans of d (8 KB apart), four K=8 steps each
#pragma unroll
          for (int span = 0; span < 4; ++span)
            mma4_tf32_ts(tS, qa[prod] + 32u * span,
                         sdesc_sw128(kb[prod] + (uint32_t)span * 8192u, 16, 1024), kIdescQK,
                         (prod > 0 || span > 0) ? 1u : 0u);
        }
        issued = true;
        tc_commit_elect(bar(kBarS));
        tc_commit_elect(bar(kBarEmpty + s));
        ++li;
      }
      // O += P_hi V_hi + P_hi V_lo + P_lo V_hi   (V stored transposed: d rows, key columns)
      {
        const uint32_t s = li % kOpSlots;
        if (!(ok = mbar_wait_warp(bar(kBarFull + s), (li / kOpSlots) & 1u, abort_flag, p.err, lim)))
          break;
        if (!(ok = mbar_wait_warp(bar(kBarP), (uint32_t)i & 1u, abort_flag, p.err, lim))) break;
        tc_fence_after();
        const uint32_t hi = sbase + s * kSlotBytes, lo = hi + kPartBytes;
        const uint32_t pa[3] = {tS, tS, tmem + kColPLo};
        const uint32_t vb[3] = {hi, lo, hi};
#pragma unroll
        for (int prod = 0; prod < 3; ++prod) {
          // two 32-key spans (16 KB apart), four K=8 steps each
#pragma unroll
          for (int span = 0; span < 2; ++span)
            mma4_tf32_ts(tO, pa[prod] + 32u * span,
                         sdesc_sw128(vb[prod] + (uint32_t)span * 16384u, 16, 1024), kIdescPV,
                         (i > 0 || prod > 0 || span > 0) ? 1u : 0u);
        }
        tc_commit_elect(bar(kBarEmpty + s));
        ++li;
      }
    }
    if (ok) tc_commit_elect(bar(kBarO));
    if (issued) {
      // everything issued must complete before TMEM is freed
      tc_commit_elect(bar(kBarDrain));
      mbar_wait_warp(bar(kBarDrain), 0, abort_flag, p.err, lim, true);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ converters
    const int cw = warp - 4;  // 0..3
    const float* kbase = p.k + (int64_t)kh * p.kv_head_stride;
    const float* vbase = p.v + (int64_t)kh * p.kv_head_stride;
    auto row_of = [&](int64_t j) -> int64_t { return p.ring_rows > 0 ? j % p.ring_rows : j; };
    bool ok = true;
    uint32_t li = 0;
    for (int i = 0; i < n && ok; ++i) {
      const int64_t key0 = (kt_first + i) * kBN;
      for (int kv = 0; kv < 2 && ok; ++kv, ++li) {
        const uint32_t s = li % kOpSlots;
        // global loads first (their latency overlaps the wait for the slot)
        float4 x[16];
        if (kv == 0) {
          // K: warp cw takes keys cw*16 .. +16; lane -> d = 4 lane
#pragma unroll
          for (int it = 0; it < 16; ++it) {
            const int64_t j = key0 + cw * 16 + it;
            x[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < L) x[it] = *reinterpret_cast<const float4*>(kbase + row_of(j) * kD + 4 * lane);
          }
        } else {
          // V: warp cw takes d = 32 cw .. +32 (quads dq = 0..7); lane -> key
          // (two halves of 32 keys)
#pragma unroll
          for (int it = 0; it < 16; ++it) {
            const int half = it >> 3, dq = it & 7;
            const int64_t j = key0 + half * 32 + lane;
            x[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < L)
              x[it] = *reinterpret_cast<const float4*>(vbase + row_of(j) * kD + 32 * cw + 4 * dq);
          }
        }
        ok = mbar_wait(bar(kBarEmpty + s), ((li / kOpSlots) & 1u) ^ 1u, abort_flag, p.err, lim);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        uint8_t* hi = smem + s * kSlotBytes;
        uint8_t* lo = hi + kPartBytes;
        if (kv == 0) {
          // K-major B tile of QK^T: 64 key rows x 128 d; 32-d spans of 128 B
          // (8 KB apart), 16-byte chunk c of row r at chunk c ^ (r & 7)
#pragma unroll
          for (int it = 0; it < 16; ++it) {
            const int r = cw * 16 + it;
            const int span = lane >> 3, c = lane & 7;
            const uint32_t off = span * 8192u + r * 128u + (uint32_t)((c ^ (r & 7)) << 4);
            const float4 v4 = x[it];
            const float4 h = make_float4(tf32_hi(v4.x), tf32_hi(v4.y), tf32_hi(v4.z), tf32_hi(v4.w));
            *reinterpret_cast<float4*>(hi + off) = h;
            *reinterpret_cast<float4*>(lo + off) =
                make_float4(v4.x - h.x, v4.y - h.y, v4.z - h.z, v4.w - h.w);
          }
        } else {
          // K-major B tile of P V: 128 d rows x 64 keys; 32-key spans of 128 B
          // (16 KB apart), key kk of row d in chunk (kk/4) ^ (d & 7), word kk%4
#pragma unroll
          for (int it = 0; it < 16; ++it) {
            const int half = it >> 3, dq = it & 7;
            const float e[4] = {x[it].x, x[it].y, x[it].z, x[it].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int d = 32 * cw + 4 * dq + q;
              const uint32_t off = half * 16384u + d * 128u +
                                   (uint32_t)((((lane >> 2) ^ (d & 7)) << 4) | ((lane & 3) << 2));
              const float h = tf32_hi(e[q]);
              *reinterpret_cast<float*>(hi + off) = h;
              *reinterpret_cast<float*>(lo + off) = e[q] - h;
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarFull + s));
      }
    }
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

    // Q row -> (hi, lo) in TMEM columns [0,128) and [128,256)
    {
      const float* qrow = p.q + t * p.qkv_dim + (int64_t)h * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t rh[32], rl[32];
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) {
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row_valid) x = *reinterpret_cast<const float4*>(qrow + c0 + 4 * v4);
          const float e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float hv = tf32_hi(e[q]);
            rh[4 * v4 + q] = __float_as_uint(hv);
            rl[4 * v4 + q] = __float_as_uint(e[q] - hv);
          }
        }
        tmem_st32(tmem + lane_off + kColQHi + c0, rh);
        tmem_st32(tmem + lane_off + kColQLo + c0, rl);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarQ));
    }

    bool ok = true;
    if (p.flags & kFlagForceTimeout) {
      // Test hook: wait on a barrier nothing signals, so the limit expires.
      ok = mbar_wait(bar(kBarDrain), 0, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    float m_run = -INFINITY, l = 0.f;
    for (int i = 0; i < n && ok; ++i) {
      ok = mbar_wait(bar(kBarS), (uint32_t)i & 1u, abort_flag, p.err, lim);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem + lane_off + kColS, r0);
      tmem_ld32(tmem + lane_off + kColS + 32, r1);
      tmem_wait_ld(r0);
      tmem_wait_ld(r1);
      float x[64];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = __uint_as_float(r0[j]) * c;
        x[32 + j] = __uint_as_float(r1[j]) * c;
      }
      const int64_t key0 = (kt_first + i) * kBN;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int64_t key = key0 + j;
        const bool vis = key <= pos && (p.window <= 0 || key > pos - p.window);
        if (!vis) x[j] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; j += 2) mx = max3f(mx, x[j], x[j + 1]);

      // Raise the exponent base only when the new maximum exceeds it by > 2^8.
      float alpha = 1.f;
      bool rescale = false;
      if (mx > m_run + kRescaleThreshold) {
        alpha = ex2(m_run - mx);  // 0 while nothing was accumulated
        rescale = (i > 0) && (m_run != -INFINITY);
        m_run = mx;
      }
      const float base = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t ph0[32], ph1[32], pl0[32], pl1[32];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float pv = ex2(x[j] - base);
        const float hv = tf32_hi(pv);
        ls[j & 3] += pv;
        if (j < 32) {
          ph0[j] = __float_as_uint(hv);
          pl0[j] = __float_as_uint(pv - hv);
        } else {
          ph1[j - 32] = __float_as_uint(hv);
          pl1[j - 32] = __float_as_uint(pv - hv);
        }
      }
      l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      // O is stable here: the commit that signalled S(i) covers P(i-1) V.
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + kColO + c0, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st32(tmem + lane_off + kColO + c0, o);
        }
      }
      tmem_st32(tmem + lane_off + kColS, ph0);
      tmem_st32(tmem + lane_off + kColS + 32, ph1);
      tmem_st32(tmem + lane_off + kColPLo, pl0);
      tmem_st32(tmem + lane_off + kColPLo + 32, pl1);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarP));
    }
    if (ok) {
      ok = mbar_wait(bar(kBarO), 0, abort_flag, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* orow = p.out + t * p.qkv_dim + (int64_t)h * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + kColO + c0, o);
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

int launch_tf32_d128(const Call& c) {
  static DeviceOnce setup;
  const int sr = setup.run(c.device, [] {
    return cudaFuncSetAttribute(tf32_d128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  tf32_d128_kernel<<<dim3((unsigned)(tiles * c.Hkv)), kThreads, kSmemAlloc, c.stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace pfa
