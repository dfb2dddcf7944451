// pfa_internal.h -- declarations shared by the C-ABI layer (pfa_api.cu) and
// the kernel translation units.  Not part of the public interface.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

namespace pfa {

// One validated call, as the launchers receive it.
struct Call {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  int64_t T, start_pos;
  int H, Hkv, D, window;
  float scale;
  cudaStream_t stream;
  unsigned* err;          // device error word of the current device
  uint64_t wait_limit_ns; // device-side wait limit
  int flags;              // kFlag* bits
  int device;
  int num_sms;
  void* ws;               // caller's workspace (device), may be null
  size_t ws_bytes;
  // Layout (defaults describe the contiguous layout of pfa_prefill_attention):
  int64_t qkv_dim;        // elements from one token's q / out row to the next (>= H*D)
  int64_t max_seq_len;    // rows per kv head in k / v (kv head stride = max_seq_len * D)
  int ring;               // 1: key j lives in row j % max_seq_len (circular cache)
  // Graph entry: device pointer to {T, start_pos}, read by the kernels at run
  // time; T above is then the largest T (the grid is sized for it).  Null
  // for every other entry point.
  const int64_t* lens;
};

// Rows at the start of each kv head's block that hold written keys: L for a
// linear cache, min(L, capacity) for a circular one.  Rows past them are
// never read (TMA reads them as zeros).
inline int64_t cache_rows_written(const Call& c) {
  if (c.lens) return c.max_seq_len;  // unknown on the host: the whole allocation
  const int64_t L = c.start_pos + c.T;
  return (c.ring && c.max_seq_len < L) ? c.max_seq_len : L;
}
// Modulus of the key -> cache row map once a circular cache has wrapped
// (L > capacity); 0 means key j is in row j.
inline int ring_rows(const Call& c) {
  if (c.lens) return c.ring ? (int)c.max_seq_len : 0;  // j % capacity == j before a wrap
  return (c.ring && c.max_seq_len < c.start_pos + c.T) ? (int)c.max_seq_len : 0;
}

constexpr int kFlagForceTimeout = 1;

// Status codes (mirror pfa_status in include/pfa.h).
constexpr int kOk = 0, kErrShape = -2, kErrDevice = -5, kErrLaunch = -6;

// One-time set-up per device (a kernel's shared-memory opt-in), safe when
// several host threads make their first call at the same time: the first
// caller runs `f` under the lock, later callers read the recorded outcome.
// Objects of this class have static storage duration (zero-initialised state).
class DeviceOnce {
 public:
  template <class F>
  int run(int device, F&& f) {
    if (device < 0 || device >= kDevices) return kErrDevice;
    int s = state_[device].load(std::memory_order_acquire);
    if (s == 0) {
      std::lock_guard<std::mutex> lk(mu_);
      s = state_[device].load(std::memory_order_relaxed);
      if (s == 0) {
        s = (f() == kOk) ? 1 : -1;
        if (s < 0) cudaGetLastError();  // clear the sticky-free error of the failed call
        state_[device].store(s, std::memory_order_release);
      }
    }
    return s > 0 ? kOk : kErrLaunch;
  }

 private:
  static constexpr int kDevices = 64;
  std::mutex mu_;
  std::atomic<int> state_[kDevices];  // 0 not done, 1 ok, -1 failed
};

// Encodes a 3-D tiled bf16 tensor map (innermost dimension first).
// Returns 0 on success.  Results are cached by all arguments.
int encode_tmap_bf16_3d(CUtensorMap* out, const void* base, const uint64_t dims[3],
                        const uint64_t strides_bytes[2], const uint32_t box[3]);

// Argument validation shared by the C entry points (pfa_api.cu): fills *c
// (without workspace) and returns a pfa_status; T == 0 gives PFA_OK with
// c->T == 0 and nothing else filled in.
int prepare(const void* q, const void* k_cache, const void* v_cache, void* out, int64_t T,
            int64_t start_pos, int num_heads, int num_kv_heads, int head_dim, int window,
            float scale, int dtype, void* stream, bool check_pointers, Call* c);
// prepare() for a caller-specified layout: q / out rows qkv_dim elements
// apart, max_seq_len rows per kv head, optionally circular (ring != 0).
int prepare_layout(const void* q, const void* k_cache, const void* v_cache, void* out,
                   int64_t T, int64_t start_pos, int num_heads, int num_kv_heads, int head_dim,
                   int window, float scale, int dtype, int64_t qkv_dim, int64_t max_seq_len,
                   int ring, void* stream, bool check_pointers, Call* c);
// Launches the kernel(s) for a prepared call (pfa_api.cu).
int dispatch(const Call& c, int dtype);

int launch_f32(const Call& c);       // fp32 on the CUDA cores, any head_dim
int launch_f32x3_d128(const Call& c); // fp32, head_dim 128, three bf16 products on the tensor cores
int launch_bf16_d128(const Call& c);
// Workspace bytes the head_dim-128 schedule the host picks needs (0: the plain
// schedule); *schedule (if not null) gets 0 plain, 1 balanced, 2 tail split.
size_t workspace_bytes_bf16_d128(const Call& c, int* schedule = nullptr);
int launch_bf16_d512(const Call& c);
// Workspace bytes of the head_dim-512 schedule the host picks (0: plain);
// *schedule (if not null) gets 0 plain or 2 tail split.
size_t workspace_bytes_bf16_d512(const Call& c, int* schedule = nullptr);
// Workspace bytes of the schedule a bf16 call gets (either head_dim).
inline size_t workspace_bytes_bf16(const Call& c, int* schedule = nullptr) {
  if (c.D == 128) return workspace_bytes_bf16_d128(c, schedule);
  if (c.D == 512) return workspace_bytes_bf16_d512(c, schedule);
  if (schedule) *schedule = 0;
  return 0;
}
// Host-only replay of the head_dim-128 work assignment with its invariants
// (pfa_debug_check_schedule); 0 or the number of the failed check.
int check_schedule_bf16_d128(const Call& c, int sms, int* schedule, int* ctas);
// The same for the head_dim-512 path (pfa_debug_check_schedule_d512).
int check_schedule_bf16_d512(const Call& c, int sms, int* schedule, int* ctas);

}  // namespace pfa
