// qkv_cte_mx_noalloc: the whole qkv_cte_mx prologue without a caller-supplied
// workspace and without any device allocation.
//
// Who needs it: host code that cannot call cudaMalloc at the point where it
// runs this operator -- for example a plugin invoked by an inference runtime
// that owns all device memory and hands its plugins no allocator, or a
// latency-critical serving loop where cudaMalloc's implicit device-wide
// synchronisation is not acceptable.  Such callers still pass their inputs and
// the output buffer; the scratch space the two kernels need (status word,
// per-token sum-of-squares partials, the per-block exponents of the Q/K codes) lives in
// the file-scope device array below.
//
// The array is part of the library image: every GPU that loads the library
// holds kNoAllocWorkspaceBytes of device memory for it until the process
// exits.  All calls share it and it keeps the last call's contents; the status
// word is cleared on every call, once every argument check has passed (the
// partials and the exponents are fully rewritten before they are read), so
// calls issued one after another are independent, but calls that overlap on the
// GPU (different streams or threads without ordering between them) race on the
// array.  A pipeline wait that runs out of time leaves its mark in the array's
// status word, which qkv_cte_mx_status reads when given a NULL workspace.
#include <mutex>

#include "rope_attention.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocWorkspaceBytes = size_t(32) << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_workspace[kNoAllocWorkspaceBytes];

std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};

}  // namespace

namespace ra {

// Device address of the array on the current device.  Host code may not use
// the symbol itself as a device pointer, so the address is looked up once per
// device (with that device current) and cached.
ra_status noalloc_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_error(RA_ERR_CUDA, "cudaGetDevice", cudaGetErrorString(e));
    return RA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_last_error(RA_ERR_INVALID_ARG, "qkv_cte_mx_noalloc", "device index out of range");
    return RA_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_dev_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess || p == nullptr) {
      set_last_error(RA_ERR_CUDA, "cudaGetSymbolAddress(static workspace)",
                     e != cudaSuccess ? cudaGetErrorString(e) : "null address");
      return RA_ERR_CUDA;
    }
    g_dev_ptr[dev] = p;
  }
  *out = g_dev_ptr[dev];
  return RA_OK;
}

}  // namespace ra

extern "C" ra_status qkv_cte_mx_noalloc(const qkv_cte_mx_params* p, const uint8_t* a,
                                        const float* a_scale, const void* w_packed,
                                        const float* weight_scales, const uint16_t* bias,
                                        const float* cos_cache, const float* sin_cache,
                                        const float* q_gamma, const float* k_gamma, uint16_t* out,
                                        void* stream) {
  return ra::qkv_cte_mx_on_library_workspace(p, a, a_scale, w_packed, weight_scales, bias, cos_cache,
                                             sin_cache, q_gamma, k_gamma, out, kNoAllocWorkspaceBytes,
                                             ra::noalloc_workspace, stream);
}
