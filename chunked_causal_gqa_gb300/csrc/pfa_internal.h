// pfa_internal.h -- declarations shared by the C-ABI layer (pfa_api.cu) and
// the kernel translation units.  Not part of the public interface.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

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
};

constexpr int kFlagForceTimeout = 1;

// Status codes (mirror pfa_status in include/pfa.h).
constexpr int kOk = 0, kErrShape = -2, kErrDevice = -5, kErrLaunch = -6;

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
// Launches the kernel(s) for a prepared call (pfa_api.cu).
int dispatch(const Call& c, int dtype);

int launch_f32(const Call& c);
int launch_bf16_d128(const Call& c);
// Workspace bytes the balanced head_dim-128 schedule needs (0: not used).
size_t workspace_bytes_bf16_d128(const Call& c);
int launch_bf16_d512(const Call& c);

}  // namespace pfa
