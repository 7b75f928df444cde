// attn_bwd_noalloc: the attention backward for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain scratch memory at the point where they
// run the backward: code that runs inside a custom allocator or memory-pool
// callback (where calling cudaMalloc would re-enter the allocator), code in
// runtimes that forbid device allocation after start-up so that memory use
// stays fixed, and plugins that receive only the input and output pointers
// from their host framework.  For them this entry point takes the same inputs
// and outputs as attn_bwd and supplies the scratch from a fixed buffer that
// lives in this file, instead of from a caller-provided workspace.
//
// The buffer is a file-scope __device__ array of ATTN_NOALLOC_SCRATCH_BYTES.
// Every GPU on which this library's code for this file is loaded holds it
// until the process exits.  Host code cannot use the array's name as a
// device address, so the first call on each device (with that device
// current) asks the runtime for the array's device address and remembers it
// for the rest of the process.  A cudaDeviceReset() makes that address stale
// (the array is placed again in the new context); the header tells callers
// not to use this entry point on a device after resetting it.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/attn_gb300.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; NULL on error.
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int attn_bwd_noalloc(void* dqkv, const void* qkv, const void* out, const void* dout, const float* lse,
                                int B, int T, int C, int NH, int NKV, float rope_theta, int dtype, void* stream) {
  const size_t need = attn_bwd_workspace_bytes(B, T, C, NH, NKV, dtype);
  if (need == 0) {
    // Invalid shape or dtype: let attn_bwd report the precise reason (it
    // validates before touching the workspace or launching anything).
    return attn_bwd(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype, nullptr, 0, stream);
  }
  if (need > (size_t)ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  void* scratch = scratch_for_current_device();
  if (scratch == nullptr) return ATTN_ERR_CUDA;
  // Nothing in the scratch has to start at zero: attn_bwd overwrites the row
  // dots and the rotated Q/K copy before reading them.
  return attn_bwd(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype, scratch,
                  (size_t)ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
