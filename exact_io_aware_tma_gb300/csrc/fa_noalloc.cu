// Backward pass without a caller-provided workspace.
//
// fa_backward needs a device workspace (LSE*log2(e), D and the fp32 dQ
// accumulator).  Some callers cannot provide one: code embedded in a host
// framework that owns every device allocation (its own pool or memory
// budget) and forbids raw cudaMalloc from plug-ins, and latency-critical
// callers that must not call cudaMalloc / cudaFree on their hot path
// because those calls can synchronise the whole device.  For them this file
// keeps the workspace in a fixed-size array of device memory that is part
// of the library image itself, so the call allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"

namespace {

// The scratch array: FA_NOALLOC_SCRATCH_BYTES of device memory, reserved on
// every GPU that loads the library and held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return FA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                                   const float* lse, const void* dout, void* dq, void* dk,
                                   void* dv, int B, int H, int N, int d, float scale, int causal,
                                   const uint8_t* block_mask, const int32_t* kv_len,
                                   void* stream) {
  // Size checks first: an invalid or too-large problem is rejected before
  // any CUDA call.
  const size_t need = fa_backward_workspace_bytes(B, H, N, d);
  if (need == 0) {
    if (d != 64 && d != 128 && B >= 1 && H >= 1 && N >= 1) return FA_ERR_UNSUPPORTED;
    return FA_ERR_INVALID_ARG;
  }
  if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  // The existing backward, handed the static array as its workspace; its
  // preprocess overwrites every part of the workspace the dK/dV/dQ kernel
  // reads (and clears the dQ accumulator), so the previous call's contents
  // never leak into this one.
  return fa_backward(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, block_mask,
                     kv_len, scratch, (size_t)FA_NOALLOC_SCRATCH_BYTES, stream);
}
