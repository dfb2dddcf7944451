// pfa_noalloc.cu -- an entry point that allocates no device memory at all.
//
// pfa_prefill_attention_ws reaches its best schedule for head_dim 128 only
// when the caller hands it a workspace, which the caller has to allocate.
// Some callers cannot: code that runs where cudaMalloc is not allowed or not
// wanted (inside a region being captured into a CUDA graph, under an
// allocator that owns all device memory and refuses foreign allocations, or
// in a host integration without a device allocator of its own).  For them,
// pfa_prefill_attention_noalloc runs the same balanced schedule with scratch
// memory that is part of this library image: a fixed array in device memory,
// created when the library's code is loaded onto a device and kept until the
// process exits.
//
// Contract (see include/pfa.h):
//  * The scratch holds at most kStaticScratchBytes.  A shape whose balanced
//    schedule needs more is refused with PFA_ERR_SCRATCH; nothing is launched.
//  * Nothing in the scratch has to start at zero: every slot a call reads was
//    written earlier by the same call.  Its contents after a call are the
//    partial results of that call.
//  * All calls on a device share the one array, so calls whose kernels can
//    overlap on the GPU (different streams without ordering between them)
//    race on it and may produce wrong results; serialise them.
//  * The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current).  Make that first call
//    outside any stream capture.
#include "pfa_internal.h"

#include "../../include/pfa.h"

#include <mutex>

namespace pfa {
namespace {

constexpr size_t kStaticScratchBytes = PFA_NOALLOC_SCRATCH_BYTES;  // per device
static_assert(kStaticScratchBytes == (size_t)32 << 20, "the header states 32 MiB");

// The scratch.  In host code this name stands for the variable, not for its
// device address: only the pointer from cudaGetSymbolAddress may reach a kernel.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64];

// Device address of the scratch on device `dev` (which must be current).
int scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= 64) return kErrDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return kErrDevice;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return kOk;
}

}  // namespace
}  // namespace pfa

using namespace pfa;

extern "C" {

int pfa_prefill_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  void* out, int64_t T, int64_t start_pos, int num_heads,
                                  int num_kv_heads, int head_dim, int window, float scale,
                                  int dtype, void* stream) {
  Call c;
  const int rc = prepare(q, k_cache, v_cache, out, T, start_pos, num_heads, num_kv_heads,
                         head_dim, window, scale, dtype, stream, true, &c);
  if (rc != PFA_OK || c.T == 0) return rc;
  if (dtype == PFA_BF16 && head_dim == 128) {
    const size_t need = workspace_bytes_bf16_d128(c);
    if (need > kStaticScratchBytes) return PFA_ERR_SCRATCH;
    if (need > 0) {
      void* scratch = nullptr;
      const int sr = scratch_address(c.device, &scratch);
      if (sr != kOk) return sr;
      c.ws = scratch;
      c.ws_bytes = kStaticScratchBytes;
    }
  }
  return dispatch(c, dtype);
}

}  // extern "C"
