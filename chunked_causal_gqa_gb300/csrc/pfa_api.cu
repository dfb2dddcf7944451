// pfa_api.cu -- the C ABI of libpfa (declared in include/pfa.h): argument
// validation, per-device state, the device error word, cached TMA tensor-map
// descriptors and kernel dispatch.
//
// The entry point follows the gate discipline of the gnosis page "Prefill
// attention -> GPU: handoff" (section "GPU design", correctness gate: any
// unsupported shape or GPU error is reported to the caller, who may fall back)
// as status codes: nothing here aborts, traps or prints unless PFA_TRACE is set.
#include "pfa_internal.h"
#include "pfa_ptx.cuh"

#include "../../include/pfa.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

namespace pfa {
namespace {

// Device-side error word (one per device context).  Kernels receive its
// address and atomically OR error bits into it.
__device__ unsigned int g_error_word;

struct DeviceState {
  bool ready = false;
  int status = kOk;       // kOk, or kErrDevice if the device is unusable
  int num_sms = 0;
  unsigned* err = nullptr;
};

std::mutex g_mutex;
DeviceState g_dev[64];
double g_wait_limit_ms = 2000.0;
int g_force_timeout = 0;

bool trace_on() {
  static const int on = [] {
    const char* e = std::getenv("PFA_TRACE");
    return (e && *e && std::strcmp(e, "0") != 0) ? 1 : 0;
  }();
  return on != 0;
}

// Per-device set-up: compute capability check, SM count, error word address.
int device_state(int* dev_out, DeviceState** st_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return kErrDevice;
  }
  std::lock_guard<std::mutex> lk(g_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return kErrDevice;
    }
    // The library is compiled for sm_103a only.
    s.status = (major == 10 && minor == 3) ? kOk : kErrDevice;
    s.num_sms = sms;
    if (s.status == kOk) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess) {
        cudaGetLastError();
        return kErrDevice;
      }
      s.err = static_cast<unsigned*>(addr);
      if (cudaMemset(s.err, 0, sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        return kErrDevice;
      }
    }
    s.ready = true;
  }
  *dev_out = dev;
  *st_out = &s;
  return s.status;
}

// A pointer the GPU can read: device memory or managed memory of this device.
bool device_accessible(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// ------------------------------------------------------------------ TMA maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (EncodeTiledFn) nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

struct MapKey {
  const void* base;
  uint64_t d0, d1, d2, s0, s1;
  uint32_t b0, b1, b2;
  bool operator==(const MapKey& o) const {
    return base == o.base && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && s0 == o.s0 &&
           s1 == o.s1 && b0 == o.b0 && b1 == o.b1 && b2 == o.b2;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base);
    const uint64_t v[8] = {k.d0, k.d1, k.d2, k.s0, k.s1, k.b0, k.b1, k.b2};
    for (uint64_t x : v) h = (h ^ x) * 0x100000001b3ull;
    return (size_t)h;
  }
};
std::mutex g_map_mutex;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

}  // namespace

int encode_tmap_bf16_3d(CUtensorMap* out, const void* base, const uint64_t dims[3],
                        const uint64_t strides_bytes[2], const uint32_t box[3]) {
  const MapKey key{base, dims[0], dims[1], dims[2], strides_bytes[0], strides_bytes[1],
                   box[0], box[1], box[2]};
  {
    std::lock_guard<std::mutex> lk(g_map_mutex);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return 0;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return -1;
  const cuuint64_t gdim[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t gstride[2] = {strides_bytes[0], strides_bytes[1]};
  const cuuint32_t bdim[3] = {box[0], box[1], box[2]};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim,
                        gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return -1;
  {
    std::lock_guard<std::mutex> lk(g_map_mutex);
    if (g_maps.size() > 1024) g_maps.clear();
    g_maps.emplace(key, m);
  }
  *out = m;
  return 0;
}

}  // namespace pfa

using namespace pfa;

extern "C" {

int pfa_version(void) { return (1 << 16) | 0; }

const char* pfa_status_string(int status) {
  switch (status) {
    case PFA_OK: return "PFA_OK";
    case PFA_ERR_NULL: return "PFA_ERR_NULL: a required pointer is NULL";
    case PFA_ERR_SHAPE: return "PFA_ERR_SHAPE: unsupported or invalid shape";
    case PFA_ERR_DTYPE: return "PFA_ERR_DTYPE: unknown dtype";
    case PFA_ERR_ALIGNMENT: return "PFA_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case PFA_ERR_DEVICE: return "PFA_ERR_DEVICE: no usable sm_103 device or pointer not on it";
    case PFA_ERR_LAUNCH: return "PFA_ERR_LAUNCH: the CUDA runtime refused the launch";
    case PFA_ERR_TIMEOUT: return "PFA_ERR_TIMEOUT: a device-side wait gave up";
    case PFA_ERR_VALUE: return "PFA_ERR_VALUE: scale is not finite";
    case PFA_ERR_ALIAS: return "PFA_ERR_ALIAS: out overlaps an input";
    case PFA_ERR_SCRATCH:
      return "PFA_ERR_SCRATCH: the shape needs more scratch than the allocation-free entry holds";
    case PFA_ERR_LENGTHS:
      return "PFA_ERR_LENGTHS: the device-side {T, start_pos} did not fit the graph call's capacities";
    default: return "PFA: unknown status";
  }
}

int pfa_debug_configure(double wait_limit_ms, int force_timeout) {
  std::lock_guard<std::mutex> lk(g_mutex);
  g_wait_limit_ms = (wait_limit_ms > 0.0) ? wait_limit_ms : 2000.0;
  g_force_timeout = force_timeout ? 1 : 0;
  return PFA_OK;
}

}  // extern "C"

namespace pfa {

// Bytes spanned by q (or out) and by each of k_cache / v_cache in a layout.
void layout_spans(int64_t T, int num_heads, int num_kv_heads, int head_dim, int dtype,
                  int64_t qkv_dim, int64_t max_seq_len, size_t* qo_bytes, size_t* kv_bytes) {
  const size_t es = dtype == PFA_F32 ? 4 : 2;
  *qo_bytes = ((size_t)(T - 1) * (size_t)qkv_dim + (size_t)num_heads * head_dim) * es;
  *kv_bytes = (size_t)num_kv_heads * (size_t)max_seq_len * head_dim * es;
}

// Validation shared by every entry point.  On success fills *c (without the
// workspace) and returns PFA_OK; T == 0 returns PFA_OK with c->T == 0.
int prepare(const void* q, const void* k_cache, const void* v_cache, void* out, int64_t T,
            int64_t start_pos, int num_heads, int num_kv_heads, int head_dim, int window,
            float scale, int dtype, void* stream, bool check_pointers, Call* c) {
  const int64_t hd = (num_heads > 0 && head_dim > 0) ? (int64_t)num_heads * head_dim : 0;
  return prepare_layout(q, k_cache, v_cache, out, T, start_pos, num_heads, num_kv_heads,
                        head_dim, window, scale, dtype, hd, start_pos + T, 0, stream,
                        check_pointers, c);
}

// The argument checks of prepare_layout that need no pointer and no CUDA
// call.  T == 0 passes once dtype, shape and scale do.
int check_args(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads, int head_dim,
               int window, float scale, int dtype, int64_t qkv_dim, int64_t max_seq_len,
               int ring) {
  if (dtype != PFA_F32 && dtype != PFA_BF16) return PFA_ERR_DTYPE;
  if (T < 0 || start_pos < 0 || num_heads <= 0 || num_kv_heads <= 0) return PFA_ERR_SHAPE;
  if (num_heads % num_kv_heads != 0) return PFA_ERR_SHAPE;
  const int group = num_heads / num_kv_heads;
  if (dtype == PFA_BF16) {
    if (head_dim != 128 && head_dim != 512) return PFA_ERR_SHAPE;
    if (group > 128) return PFA_ERR_SHAPE;
  } else {
    if (head_dim <= 0 || head_dim > 512 || head_dim % 4 != 0) return PFA_ERR_SHAPE;
  }
  const int64_t L = start_pos + T;
  // TMA coordinates and launch indices are 32-bit.
  if (L > ((int64_t)1 << 31) - 4096 || T > ((int64_t)1 << 31) - 4096) return PFA_ERR_SHAPE;
  if (!std::isfinite(scale)) return PFA_ERR_VALUE;
  if (T == 0) return PFA_OK;
  // ---- layout
  if (qkv_dim < (int64_t)num_heads * head_dim || max_seq_len <= 0 ||
      max_seq_len > ((int64_t)1 << 31) - 4096)
    return PFA_ERR_SHAPE;
  if (!ring && max_seq_len < L) return PFA_ERR_SHAPE;
  if (ring) {
    // every key some row of the chunk sees must still be in the cache
    if (window <= 0) return PFA_ERR_SHAPE;
    const int64_t span = std::min<int64_t>(L, (int64_t)window + T - 1);
    if (max_seq_len < span) return PFA_ERR_SHAPE;
    // a wrapped bf16 ring must not wrap inside a 128-key tile
    if (dtype == PFA_BF16 && max_seq_len < L && max_seq_len % 128 != 0) return PFA_ERR_SHAPE;
  }
  if ((qkv_dim * (dtype == PFA_F32 ? 4 : 2)) % 16 != 0) return PFA_ERR_ALIGNMENT;
  return PFA_OK;
}

int prepare_layout(const void* q, const void* k_cache, const void* v_cache, void* out,
                   int64_t T, int64_t start_pos, int num_heads, int num_kv_heads, int head_dim,
                   int window, float scale, int dtype, int64_t qkv_dim, int64_t max_seq_len,
                   int ring, void* stream, bool check_pointers, Call* c) {
  // ---- pure argument checks (no CUDA calls)
  const int ac = check_args(T, start_pos, num_heads, num_kv_heads, head_dim, window, scale,
                            dtype, qkv_dim, max_seq_len, ring);
  if (ac != PFA_OK) return ac;
  c->T = T;
  if (T == 0) return PFA_OK;
  if (check_pointers) {
    if (!q || !k_cache || !v_cache || !out) return PFA_ERR_NULL;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                          reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out);
    if (mis & 15u) return PFA_ERR_ALIGNMENT;
    size_t qo_bytes = 0, kv_bytes = 0;
    layout_spans(T, num_heads, num_kv_heads, head_dim, dtype, qkv_dim, max_seq_len, &qo_bytes,
                 &kv_bytes);
    if (overlaps(out, qo_bytes, q, qo_bytes) || overlaps(out, qo_bytes, k_cache, kv_bytes) ||
        overlaps(out, qo_bytes, v_cache, kv_bytes))
      return PFA_ERR_ALIAS;
  }

  // ---- device checks
  int dev = -1;
  DeviceState* st = nullptr;
  const int ds = device_state(&dev, &st);
  if (ds != kOk) return ds;
  if (check_pointers &&
      (!device_accessible(q, dev) || !device_accessible(k_cache, dev) ||
       !device_accessible(v_cache, dev) || !device_accessible(out, dev)))
    return PFA_ERR_DEVICE;

  c->q = q;
  c->k = k_cache;
  c->v = v_cache;
  c->out = out;
  c->start_pos = start_pos;
  c->H = num_heads;
  c->Hkv = num_kv_heads;
  c->D = head_dim;
  c->window = window > 0 ? window : 0;
  c->scale = scale;
  c->stream = static_cast<cudaStream_t>(stream);
  c->err = st->err;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    c->wait_limit_ns = (uint64_t)(g_wait_limit_ms * 1e6);
    c->flags = g_force_timeout ? kFlagForceTimeout : 0;
  }
  c->device = dev;
  c->num_sms = st->num_sms;
  c->ws = nullptr;
  c->ws_bytes = 0;
  c->qkv_dim = qkv_dim;
  c->max_seq_len = max_seq_len;
  c->ring = ring ? 1 : 0;
  c->lens = nullptr;
  return PFA_OK;
}

// Attaches a caller workspace to a prepared call after checking it.
int attach_workspace(Call* c, int dtype, void* workspace, size_t workspace_bytes) {
  if (workspace == nullptr || workspace_bytes == 0) return PFA_OK;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PFA_ERR_ALIGNMENT;
  if (!device_accessible(workspace, c->device)) return PFA_ERR_DEVICE;
  size_t qo_bytes = 0, kv_bytes = 0;
  layout_spans(c->T, c->H, c->Hkv, c->D, dtype, c->qkv_dim, c->max_seq_len, &qo_bytes,
               &kv_bytes);
  if (overlaps(workspace, workspace_bytes, c->out, qo_bytes) ||
      overlaps(workspace, workspace_bytes, c->q, qo_bytes) ||
      overlaps(workspace, workspace_bytes, c->k, kv_bytes) ||
      overlaps(workspace, workspace_bytes, c->v, kv_bytes))
    return PFA_ERR_ALIAS;
  c->ws = workspace;
  c->ws_bytes = workspace_bytes;
  return PFA_OK;
}

int dispatch(const Call& c, int dtype) {
  int rc;
  if (dtype == PFA_F32)
    // the tensor-core kernel packs a GQA group into 128-row tiles (group <= 128)
    rc = (c.D == 128 && c.H / c.Hkv <= 128) ? launch_f32x3_d128(c) : launch_f32(c);
  else if (c.D == 128)
    rc = launch_bf16_d128(c);
  else
    rc = launch_bf16_d512(c);
  if (trace_on())
    std::fprintf(stderr,
                 "[pfa] dtype=%d T=%lld start_pos=%lld H=%d Hkv=%d D=%d window=%d ws=%zu -> %d\n",
                 dtype, (long long)c.T, (long long)c.start_pos, c.H, c.Hkv, c.D, c.window,
                 c.ws_bytes, rc);
  return rc;
}

// ------------------------------------------------------------------ host-buffer entry
namespace {

constexpr int kHostGroups = 4;  // most kv-head groups of pfa_prefill_attention_host

// Groups for a call moving `bytes` between host and device: one below 4 MiB
// (the copies are too short to overlap), two below 128 MiB, else four --
// the fastest of 1, 2 and 4 measured on GB300 for a 1.3 MB fp32 layer, the
// 28 MB Mistral-shaped layer, the 46-67 MB head_dim-512 layers and the
// 294 MB 64k chunk.
int host_groups(size_t bytes, int num_kv_heads) {
  const int g = bytes < ((size_t)4 << 20) ? 1 : (bytes < ((size_t)128 << 20) ? 2 : kHostGroups);
  return std::min(g, num_kv_heads);
}

// Streams and events of the host-buffer entry on one device, created on the
// first call there and kept until the process exits.
struct HostPipe {
  cudaStream_t s[kHostGroups];
  cudaEvent_t fork;                  // the caller's stream reached the call
  cudaEvent_t in_done[kHostGroups];  // group g's inputs are on the device
  cudaEvent_t done[kHostGroups];     // group g's output is back in host memory
};
std::mutex g_host_mutex;  // held while a call enqueues its work
HostPipe* g_host_pipe[64];

int host_pipe(int dev, HostPipe** out) {
  if (dev < 0 || dev >= 64) return kErrDevice;
  if (!g_host_pipe[dev]) {
    HostPipe hp;
    bool ok = cudaEventCreateWithFlags(&hp.fork, cudaEventDisableTiming) == cudaSuccess;
    for (int g = 0; g < kHostGroups && ok; ++g)
      ok = cudaStreamCreateWithFlags(&hp.s[g], cudaStreamNonBlocking) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.in_done[g], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.done[g], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return kErrDevice;
    }
    g_host_pipe[dev] = new HostPipe(hp);
  }
  *out = g_host_pipe[dev];
  return kOk;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// The host entry's work split and device buffer for a prepared call c0 (the
// contiguous layout): the device copies of q, k, v and out at off[0..3],
// then one workspace per group of kv heads (the schedule
// pfa_prefill_attention_ws picks for the group's heads alone; groups run
// at the same time, so each has its own).
struct HostPlan {
  int G;                          // groups; group g has kv heads [a[g], a[g+1])
  int a[kHostGroups + 1];
  size_t off[4];
  size_t ws_off[kHostGroups], ws_len[kHostGroups];
  size_t total;                   // bytes of the device buffer
};

void host_plan(const Call& c0, int dtype, HostPlan* hp) {
  const size_t es = dtype == PFA_F32 ? 4 : 2;
  const int64_t L = c0.start_pos + c0.T;
  const size_t qo = (size_t)c0.T * c0.H * c0.D * es, kv = (size_t)c0.Hkv * L * c0.D * es;
  hp->off[0] = 0;
  hp->off[1] = round256(qo);
  hp->off[2] = hp->off[1] + round256(kv);
  hp->off[3] = hp->off[2] + round256(kv);
  size_t at = hp->off[3] + round256(qo);
  hp->G = host_groups(2 * qo + 2 * kv, c0.Hkv);
  const int group = c0.H / c0.Hkv;
  for (int g = 0; g <= hp->G; ++g) hp->a[g] = g * c0.Hkv / hp->G;
  for (int g = 0; g < hp->G; ++g) {
    size_t need = 0;
    if (dtype == PFA_BF16) {
      Call cg = c0;
      cg.Hkv = hp->a[g + 1] - hp->a[g];
      cg.H = cg.Hkv * group;
      need = workspace_bytes_bf16(cg);
    }
    hp->ws_off[g] = at;
    hp->ws_len[g] = need;
    at += round256(need);
  }
  hp->total = at;
}

// A T x width-byte block of rows `pitch` bytes apart (one copy when the rows
// are contiguous).
cudaError_t copy_rows(void* dst, const void* src, size_t pitch, size_t width, int64_t T,
                      cudaStream_t s) {
  if (width == pitch) return cudaMemcpyAsync(dst, src, (size_t)T * pitch, cudaMemcpyDefault, s);
  return cudaMemcpy2DAsync(dst, pitch, src, pitch, width, (size_t)T, cudaMemcpyDefault, s);
}

}  // namespace

}  // namespace pfa

extern "C" {

int pfa_prefill_attention(const void* q, const void* k_cache, const void* v_cache, void* out,
                          int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                          int head_dim, int window, float scale, int dtype, void* stream) {
  return pfa_prefill_attention_ws(q, k_cache, v_cache, out, T, start_pos, num_heads,
                                  num_kv_heads, head_dim, window, scale, dtype, nullptr, 0,
                                  stream);
}

int pfa_prefill_attention_ws(const void* q, const void* k_cache, const void* v_cache, void* out,
                             int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                             int head_dim, int window, float scale, int dtype, void* workspace,
                             size_t workspace_bytes, void* stream) {
  Call c;
  int rc = prepare(q, k_cache, v_cache, out, T, start_pos, num_heads, num_kv_heads, head_dim,
                   window, scale, dtype, stream, true, &c);
  if (rc != PFA_OK || c.T == 0) return rc;
  if ((rc = attach_workspace(&c, dtype, workspace, workspace_bytes)) != PFA_OK) return rc;
  return dispatch(c, dtype);
}

int pfa_prefill_attention_cache(const void* q, const void* k_cache, const void* v_cache,
                                void* out, int64_t T, int64_t start_pos, int num_heads,
                                int num_kv_heads, int head_dim, int window, float scale,
                                int dtype, int64_t qkv_dim, int64_t max_seq_len, int ring,
                                void* workspace, size_t workspace_bytes, void* stream) {
  Call c;
  int rc = prepare_layout(q, k_cache, v_cache, out, T, start_pos, num_heads, num_kv_heads,
                          head_dim, window, scale, dtype, qkv_dim, max_seq_len, ring, stream,
                          true, &c);
  if (rc != PFA_OK || c.T == 0) return rc;
  if ((rc = attach_workspace(&c, dtype, workspace, workspace_bytes)) != PFA_OK) return rc;
  return dispatch(c, dtype);
}

int pfa_prefill_attention_graph(const void* q, const void* k_cache, const void* v_cache,
                                void* out, const int64_t* lengths, int64_t max_T,
                                int num_heads, int num_kv_heads, int head_dim, int window,
                                float scale, int dtype, int64_t qkv_dim, int64_t max_seq_len,
                                int ring, void* stream) {
  if (!lengths) return PFA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(lengths) & 7u) return PFA_ERR_ALIGNMENT;
  // The host knows only the capacities: validate as a chunk of max_T tokens
  // at position 0 (so max_T <= max_seq_len); the kernels check the run-time
  // values against the same limits.
  Call c;
  const int rc = prepare_layout(q, k_cache, v_cache, out, max_T, 0, num_heads, num_kv_heads,
                                head_dim, window, scale, dtype, qkv_dim, max_seq_len, ring,
                                stream, true, &c);
  if (rc != PFA_OK || c.T == 0) return rc;
  // a bf16 ring may wrap at run time: it must wrap on 128-key tile boundaries
  if (ring && dtype == PFA_BF16 && max_seq_len % 128 != 0) return PFA_ERR_SHAPE;
  if (!device_accessible(lengths, c.device)) return PFA_ERR_DEVICE;
  c.lens = lengths;
  return dispatch(c, dtype);
}

int pfa_workspace_bytes(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                        int head_dim, int window, int dtype, size_t* bytes) {
  if (!bytes) return PFA_ERR_NULL;
  *bytes = 0;
  Call c;
  const int rc = prepare(nullptr, nullptr, nullptr, nullptr, T, start_pos, num_heads,
                         num_kv_heads, head_dim, window, 1.0f, dtype, nullptr, false, &c);
  if (rc != PFA_OK || c.T == 0) return rc;
  if (dtype == PFA_BF16) *bytes = workspace_bytes_bf16(c);
  return PFA_OK;
}

int pfa_schedule(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads, int head_dim,
                 int window, int dtype, int* schedule, size_t* workspace_bytes) {
  if (!schedule || !workspace_bytes) return PFA_ERR_NULL;
  *schedule = PFA_SCHEDULE_PLAIN;
  *workspace_bytes = 0;
  Call c;
  const int rc = prepare(nullptr, nullptr, nullptr, nullptr, T, start_pos, num_heads,
                         num_kv_heads, head_dim, window, 1.0f, dtype, nullptr, false, &c);
  if (rc != PFA_OK || c.T == 0) return rc;
  if (dtype == PFA_BF16) *workspace_bytes = workspace_bytes_bf16(c, schedule);
  return PFA_OK;
}

int pfa_debug_check_schedule(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                             int window, int num_sms, int* schedule, int* ctas,
                             int* failed_check) {
  if (!schedule || !ctas || !failed_check) return PFA_ERR_NULL;
  *schedule = 0;
  *ctas = 0;
  *failed_check = 0;
  if (num_sms <= 0 || num_sms > 1024) return PFA_ERR_SHAPE;
  // shape checks of the bf16 head_dim-128 path, without a device
  if (T < 0 || start_pos < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || num_heads / num_kv_heads > 128)
    return PFA_ERR_SHAPE;
  const int64_t L = start_pos + T;
  if (L > ((int64_t)1 << 31) - 4096) return PFA_ERR_SHAPE;
  if (T == 0) return PFA_OK;
  Call c{};
  c.T = T;
  c.start_pos = start_pos;
  c.H = num_heads;
  c.Hkv = num_kv_heads;
  c.D = 128;
  c.window = window > 0 ? window : 0;
  c.qkv_dim = (int64_t)num_heads * 128;
  c.max_seq_len = L;
  *failed_check = check_schedule_bf16_d128(c, num_sms, schedule, ctas);
  return PFA_OK;
}

int pfa_debug_check_schedule_d512(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                                  int window, int num_sms, int* schedule, int* ctas,
                                  int* failed_check) {
  if (!schedule || !ctas || !failed_check) return PFA_ERR_NULL;
  *schedule = 0;
  *ctas = 0;
  *failed_check = 0;
  if (num_sms <= 0 || num_sms > 1024) return PFA_ERR_SHAPE;
  // shape checks of the bf16 head_dim-512 path, without a device
  if (T < 0 || start_pos < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || num_heads / num_kv_heads > 128)
    return PFA_ERR_SHAPE;
  const int64_t L = start_pos + T;
  if (L > ((int64_t)1 << 31) - 4096) return PFA_ERR_SHAPE;
  if (T == 0) return PFA_OK;
  Call c{};
  c.T = T;
  c.start_pos = start_pos;
  c.H = num_heads;
  c.Hkv = num_kv_heads;
  c.D = 512;
  c.window = window > 0 ? window : 0;
  c.qkv_dim = (int64_t)num_heads * 512;
  c.max_seq_len = L;
  *failed_check = check_schedule_bf16_d512(c, num_sms, schedule, ctas);
  return PFA_OK;
}

int pfa_host_buffer_bytes(int64_t T, int64_t start_pos, int num_heads, int num_kv_heads,
                          int head_dim, int window, int dtype, size_t* bytes) {
  if (!bytes) return PFA_ERR_NULL;
  *bytes = 0;
  Call c;
  const int rc = prepare(nullptr, nullptr, nullptr, nullptr, T, start_pos, num_heads,
                         num_kv_heads, head_dim, window, 1.0f, dtype, nullptr, false, &c);
  if (rc != PFA_OK || c.T == 0) return rc;
  HostPlan hp;
  host_plan(c, dtype, &hp);
  *bytes = hp.total;
  return PFA_OK;
}

int pfa_prefill_attention_host(const void* q, const void* k_cache, const void* v_cache,
                               void* out, int64_t T, int64_t start_pos, int num_heads,
                               int num_kv_heads, int head_dim, int window, float scale,
                               int dtype, void* device_buffer, size_t device_buffer_bytes,
                               void* stream) {
  // argument checks before any CUDA call, in the order of pfa_prefill_attention
  const int64_t L = start_pos + T;
  int rc = check_args(T, start_pos, num_heads, num_kv_heads, head_dim, window, scale, dtype,
                      (int64_t)num_heads * head_dim, L, 0);
  if (rc != PFA_OK || T == 0) return rc;
  if (!q || !k_cache || !v_cache || !out || !device_buffer) return PFA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return PFA_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(device_buffer) & 255u) return PFA_ERR_ALIGNMENT;
  const size_t es = dtype == PFA_F32 ? 4 : 2;
  const size_t row = (size_t)num_heads * head_dim * es;     // a token's q / out row
  const size_t head_kv = (size_t)L * head_dim * es;         // a kv head's K (or V) block
  const size_t qo = (size_t)T * row, kv = (size_t)num_kv_heads * head_kv;
  if (overlaps(out, qo, q, qo) || overlaps(out, qo, k_cache, kv) || overlaps(out, qo, v_cache, kv))
    return PFA_ERR_ALIAS;
  // device checks, then the split and the buffer it needs
  Call c0;
  rc = prepare(nullptr, nullptr, nullptr, nullptr, T, start_pos, num_heads, num_kv_heads,
               head_dim, window, scale, dtype, stream, false, &c0);
  if (rc != PFA_OK) return rc;
  HostPlan plan;
  host_plan(c0, dtype, &plan);
  if (device_buffer_bytes < plan.total) return PFA_ERR_SHAPE;
  if (overlaps(device_buffer, plan.total, q, qo) || overlaps(device_buffer, plan.total, k_cache, kv) ||
      overlaps(device_buffer, plan.total, v_cache, kv) ||
      overlaps(device_buffer, plan.total, out, qo))
    return PFA_ERR_ALIAS;
  if (!device_accessible(device_buffer, c0.device)) return PFA_ERR_DEVICE;

  // One call per group of kv heads on the device copies: q / out rows keep
  // the full row pitch (qkv_dim = H * D), K / V point at the group's heads.
  char* base = static_cast<char*>(device_buffer);
  char *qd = base + plan.off[0], *kd = base + plan.off[1], *vd = base + plan.off[2],
       *od = base + plan.off[3];
  const int group = num_heads / num_kv_heads;
  const int G = plan.G;
  Call gc[kHostGroups];
  size_t col[kHostGroups], width[kHostGroups], kvoff[kHostGroups], kvlen[kHostGroups];
  for (int g = 0; g < G; ++g) {
    const int a = plan.a[g], b = plan.a[g + 1];
    col[g] = (size_t)a * group * head_dim * es;
    width[g] = (size_t)(b - a) * group * head_dim * es;
    kvoff[g] = (size_t)a * head_kv;
    kvlen[g] = (size_t)(b - a) * head_kv;
    // the group's pointers lie inside the device buffer checked above
    rc = prepare_layout(qd + col[g], kd + kvoff[g], vd + kvoff[g], od + col[g], T, start_pos,
                        (b - a) * group, b - a, head_dim, window, scale, dtype,
                        (int64_t)num_heads * head_dim, L, 0, nullptr, false, &gc[g]);
    if (rc != PFA_OK) return rc;
    if (plan.ws_len[g] > 0) {
      gc[g].ws = base + plan.ws_off[g];
      gc[g].ws_bytes = plan.ws_len[g];
    }
  }

  std::lock_guard<std::mutex> lk(g_host_mutex);
  HostPipe* hp = nullptr;
  if ((rc = host_pipe(c0.device, &hp)) != kOk) return rc;
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  if (cudaEventRecord(hp->fork, user) != cudaSuccess) {
    cudaGetLastError();
    return PFA_ERR_LAUNCH;
  }
  int status = PFA_OK;
  int joined = 0;  // groups whose work `stream` must wait for
  for (int g = 0; g < G && status == PFA_OK; ++g) {
    cudaStream_t s = hp->s[g];
    bool ok = cudaStreamWaitEvent(s, hp->fork, 0) == cudaSuccess &&
              (g == 0 || cudaStreamWaitEvent(s, hp->in_done[g - 1], 0) == cudaSuccess);
    // inputs: the group's K and V blocks and its q columns, groups in order
    ok = ok &&
         cudaMemcpyAsync(kd + kvoff[g], static_cast<const char*>(k_cache) + kvoff[g], kvlen[g],
                         cudaMemcpyDefault, s) == cudaSuccess &&
         cudaMemcpyAsync(vd + kvoff[g], static_cast<const char*>(v_cache) + kvoff[g], kvlen[g],
                         cudaMemcpyDefault, s) == cudaSuccess &&
         copy_rows(qd + col[g], static_cast<const char*>(q) + col[g], row, width[g], T, s) ==
             cudaSuccess &&
         cudaEventRecord(hp->in_done[g], s) == cudaSuccess;
    if (ok) {
      gc[g].stream = s;
      status = dispatch(gc[g], dtype);
      ok = status == PFA_OK &&
           copy_rows(static_cast<char*>(out) + col[g], od + col[g], row, width[g], T, s) ==
               cudaSuccess;
    }
    // whatever was queued on s is joined back into the caller's stream
    if (cudaEventRecord(hp->done[g], s) == cudaSuccess) joined = g + 1;
    if (!ok && status == PFA_OK) status = PFA_ERR_LAUNCH;
  }
  for (int g = 0; g < joined; ++g)
    if (cudaStreamWaitEvent(user, hp->done[g], 0) != cudaSuccess && status == PFA_OK)
      status = PFA_ERR_LAUNCH;
  if (status != PFA_OK) cudaGetLastError();
  return status;
}

int pfa_last_device_error(void* stream) {
  int dev = -1;
  DeviceState* st = nullptr;
  const int ds = device_state(&dev, &st);
  if (ds != kOk) return ds;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return PFA_ERR_DEVICE;
  }
  unsigned word = 0;
  if (cudaMemcpyAsync(&word, st->err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(st->err, 0, sizeof(unsigned), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return PFA_ERR_DEVICE;
  }
  if (word & kErrTimeout) return PFA_ERR_TIMEOUT;
  if (word & kErrLengths) return PFA_ERR_LENGTHS;
  return PFA_OK;
}

}  // extern "C"
