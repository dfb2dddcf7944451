// pfa_f32.cu -- fp32 prefill attention on the CUDA cores (exact fp32 FMA).
//
// Serves the fp32 dtype, whose accuracy bar is max |gpu - fp64| <= 1e-4 (the
// bar of the gnosis page "Prefill attention -> GPU: handoff", section
// "Implementation status", GPU-vs-CPU parity).  The tensor cores' tf32 mode
// keeps only 10 mantissa bits, so this path stays on fp32 FMAs.
//
// Work decomposition: a block owns one kv head and 8 consecutive rows of that
// head's token-major row set (row r -> token r / group, query head
// kv_head * group + r % group), one warp per row, so every K/V tile staged in
// shared memory is read by all query heads of the GQA group.  Keys stream in
// tiles of 32: lane j scores key j of the tile (a full dot product against the
// warp's query row), the warp takes the tile maximum and sum with shuffles,
// updates its online-softmax state and accumulates P.V with each lane owning
// head_dim / 32 output columns.  head_dim is a multiple of 4, so every row is
// 16-byte aligned and moves as float4 vectors.  The causal / window mask is
// evaluated from the indices; no mask tensor exists.
#include "pfa_internal.h"
#include "pfa_ptx.cuh"

#include <cmath>

namespace pfa {
namespace {

constexpr int kRowsPerBlock = 8;      // one warp per row
constexpr int kKeysPerTile = 32;
constexpr int kMaxD = 512;
constexpr int kMaxCols = kMaxD / 32;  // output columns per lane
constexpr int kLoadBatch = 4;         // float4 loads in flight per thread and tensor

struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  int64_t q_stride;        // elements from one token's q / out row to the next
  int64_t kv_head_stride;  // elements from one kv head's cache block to the next
  int64_t ring_rows;       // > 0: key j is in cache row j % ring_rows; 0: in row j
  int64_t T, start_pos, L;  // graph entry: T = the largest T, start_pos unused
  const int64_t* lens;      // graph entry: device {T, start_pos}; else null
  int64_t kv_capacity;      // rows per kv head in the cache
  unsigned* err;            // device error word
  int H, Hkv, group, D, window;
  float scale_log2;        // scale * log2(e)
  int64_t rows_per_head;   // T * group
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(kRowsPerBlock * 32)
f32_attention_kernel(const F32Params p) {
  extern __shared__ float smem[];
  const int D = p.D;
  // K rows padded by 4 floats: lane j's 16-byte reads of row j fall in a
  // distinct quarter of the banks for every 8 consecutive lanes.
  const int Dp = D + 4;
  float* sK = smem;                            // [32][D+4]
  float* sV = sK + kKeysPerTile * Dp;          // [32][D]
  float* sQ = sV + kKeysPerTile * D;           // [8][D]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Chunk length and position: kernel parameters, or (graph entry) read from
  // device memory at run time, with the grid sized for the largest T.
  int64_t start_pos = p.start_pos, rows_per_head = p.rows_per_head;
  if (p.lens) {
    const int64_t T = p.lens[0];
    start_pos = p.lens[1];
    if (!lengths_ok(T, start_pos, p.T, p.kv_capacity, p.ring_rows, p.window)) {
      if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(p.err, kErrLengths);
      return;
    }
    rows_per_head = T * p.group;
  }
  const int kh = blockIdx.y;
  const int64_t r0 = (int64_t)blockIdx.x * kRowsPerBlock;
  if (r0 >= rows_per_head) return;  // the whole block (graph entry, shorter chunk)
  const int64_t r = r0 + warp;
  const bool active = r < rows_per_head;
  const int64_t t = active ? r / p.group : 0;
  const int h = kh * p.group + (active ? (int)(r % p.group) : 0);
  const int64_t pos = start_pos + t;

  for (int d = lane; d < D; d += 32)
    sQ[warp * D + d] = active ? p.q[t * p.q_stride + h * (int64_t)D + d] : 0.f;

  // Keys any row of this block can see.
  const int64_t r_last = min(r0 + kRowsPerBlock, rows_per_head) - 1;
  const int64_t pos_lo = start_pos + r0 / p.group;
  const int64_t pos_hi = start_pos + r_last / p.group;
  const int64_t kmin = p.window > 0 ? max((int64_t)0, pos_lo - p.window + 1) : 0;
  const int64_t kmax = pos_hi;

  const float* kbase = p.k + (int64_t)kh * p.kv_head_stride;
  const float* vbase = p.v + (int64_t)kh * p.kv_head_stride;
  const int ncols = (D + 31) >> 5;

  float m = -INFINITY, l = 0.f;
  float o[kMaxCols];
#pragma unroll
  for (int c = 0; c < kMaxCols; ++c) o[c] = 0.f;

  for (int64_t j0 = kmin; j0 <= kmax; j0 += kKeysPerTile) {
    __syncthreads();  // previous tile fully consumed (and sQ written, first pass)
    // 4-float vectors; up to kLoadBatch vectors of K and of V per thread are
    // loaded into registers before any is stored, so their DRAM latencies overlap.
    const int nvec = kKeysPerTile * D / 4;
    for (int base = threadIdx.x; base < nvec; base += kLoadBatch * blockDim.x) {
      float4 kr4[kLoadBatch], vr4[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int idx = base + u * blockDim.x;
        kr4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        vr4[u] = kr4[u];
        if (idx < nvec) {
          const int jj = (idx * 4) / D;
          const int64_t j = j0 + jj;
          if (j <= kmax) {
            const int d = idx * 4 - jj * D;
            const int64_t row = p.ring_rows > 0 ? j % p.ring_rows : j;
            kr4[u] = *reinterpret_cast<const float4*>(kbase + row * D + d);
            vr4[u] = *reinterpret_cast<const float4*>(vbase + row * D + d);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int idx = base + u * blockDim.x;
        if (idx < nvec) {
          const int jj = (idx * 4) / D, d = idx * 4 - jj * D;
          *reinterpret_cast<float4*>(sK + jj * Dp + d) = kr4[u];
          *reinterpret_cast<float4*>(sV + jj * D + d) = vr4[u];
        }
      }
    }
    __syncthreads();

    // lane scores key j0 + lane
    const int64_t j = j0 + lane;
    const float4* qr = reinterpret_cast<const float4*>(sQ + warp * D);
    const float4* kr = reinterpret_cast<const float4*>(sK + lane * Dp);
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;   // four independent chains
#pragma unroll 4
    for (int d4 = 0; d4 < D / 4; ++d4) {
      const float4 a = qr[d4], b = kr[d4];
      s0 = fmaf(a.x, b.x, s0);
      s1 = fmaf(a.y, b.y, s1);
      s2 = fmaf(a.z, b.z, s2);
      s3 = fmaf(a.w, b.w, s3);
    }
    const float s = (s0 + s1) + (s2 + s3);
    const bool vis = active && j <= pos && (p.window <= 0 || j > pos - p.window);
    const float x = vis ? s * p.scale_log2 : -INFINITY;

    const float m_new = fmaxf(m, warp_max(x));
    const float base = (m_new == -INFINITY) ? 0.f : m_new;   // no visible key yet
    const float alpha = ex2(m - base);                        // 0 when m = -inf
    const float pj = ex2(x - base);
    l = l * alpha + warp_sum(pj);
#pragma unroll
    for (int c = 0; c < kMaxCols; ++c) o[c] *= alpha;
    for (int jj = 0; jj < kKeysPerTile; ++jj) {
      const float pb = __shfl_sync(0xffffffffu, pj, jj);
      const float* vr = sV + jj * D;
#pragma unroll
      for (int c = 0; c < kMaxCols; ++c) {
        const int d = lane + 32 * c;
        if (c < ncols && d < D) o[c] = fmaf(pb, vr[d], o[c]);
      }
    }
    m = m_new;
  }

  if (active) {
    const float inv = 1.f / l;
    float* orow = p.out + t * p.q_stride + h * (int64_t)D;
#pragma unroll
    for (int c = 0; c < kMaxCols; ++c) {
      const int d = lane + 32 * c;
      if (c < ncols && d < D) orow[d] = o[c] * inv;
    }
  }
}

size_t smem_bytes(int D) {
  return sizeof(float) * ((size_t)kKeysPerTile * (D + 4) + (size_t)kKeysPerTile * D +
                          (size_t)kRowsPerBlock * D);
}

}  // namespace

int launch_f32(const Call& c) {
  static DeviceOnce setup;
  const int sr = setup.run(c.device, [] {
    return cudaFuncSetAttribute(f32_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes(kMaxD)) == cudaSuccess ? kOk : kErrLaunch;
  });
  if (sr != kOk) return sr;
  const size_t smem = smem_bytes(c.D);
  F32Params p;
  p.q = static_cast<const float*>(c.q);
  p.k = static_cast<const float*>(c.k);
  p.v = static_cast<const float*>(c.v);
  p.out = static_cast<float*>(c.out);
  p.q_stride = c.qkv_dim;
  p.kv_head_stride = c.max_seq_len * (int64_t)c.D;
  p.ring_rows = ring_rows(c);
  p.lens = c.lens;
  p.kv_capacity = c.max_seq_len;
  p.err = c.err;
  p.T = c.T;
  p.start_pos = c.start_pos;
  p.L = c.start_pos + c.T;
  p.H = c.H;
  p.Hkv = c.Hkv;
  p.group = c.H / c.Hkv;
  p.D = c.D;
  p.window = c.window;
  p.scale_log2 = (float)((double)c.scale * 1.4426950408889634);
  p.rows_per_head = c.T * (int64_t)p.group;
  const int64_t bx = (p.rows_per_head + kRowsPerBlock - 1) / kRowsPerBlock;
  if (bx > 0x7fffffff || c.Hkv > 65535) return kErrShape;
  dim3 grid((unsigned)bx, (unsigned)c.Hkv);
  f32_attention_kernel<<<grid, kRowsPerBlock * 32, smem, c.stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace pfa
