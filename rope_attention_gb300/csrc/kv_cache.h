// Internal interface of the KvRmsNormRopeCache kernel (kv_cache.cu) for the C-ABI layer.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ra {

// quantised cache element types (0 = not quantised: the input dtype)
enum KvQuant : int32_t { kQuantNone = 0, kQuantInt8 = 1, kQuantE4m3 = 2, kQuantE5m2 = 3 };
// cache modes, numbered as RA_CACHE_* in the public header
enum KvMode : int32_t { kModeNorm = 0, kModePa = 1, kModePaBnsd = 2, kModePaBlkBnsd = 4 };

struct KvLaunch {
  const uint16_t* kv;          // bf16 or fp16 bit patterns (f16 below), like gamma/cos/sin/v
  const uint16_t* gamma;
  const uint16_t* cos;
  const uint16_t* sin;
  const int64_t* index;
  void* k_cache;
  void* ckv_cache;
  const float* k_scale;
  const float* k_offset;
  const float* v_scale;
  const float* v_offset;
  const uint16_t* v;
  uint16_t* k_rope;
  uint16_t* c_kv;
  int32_t* err_count;
  int32_t* status;             // kv_status_word(); the staged kernel runs only when it is known
  int64_t B, N, S, Dkv, Dv;
  int32_t R;                   // rope size
  int32_t variant;             // 1 or 2
  int32_t mode;                // KvMode
  int64_t block_num, block_size;
  int64_t cache_seq;           // Norm mode: Scache
  float eps;
  int32_t out_kv;              // write k_rope / c_kv
  int32_t f16;                 // inputs (and unquantised caches, outputs) are fp16
  int32_t kq, vq;              // KvQuant of the k / ckv cache
  int32_t k_scalar, v_scalar;  // V1: the component's scale / offset are one value [1]
  int32_t rope_bcast;          // cos/sin are [B, N, 1, R]
  int64_t wait_ns;             // time limit of each pipeline wait (staged kernel)
  int32_t stall_loads;         // test hook: the staged kernel issues no copies, so its waits run out
};
// Device address of this library's KV status word on the current device (0 = fine,
// 1 = a pipeline wait of the staged kernel gave up); nullptr if it cannot be found.
int32_t* kv_status_word();
cudaError_t launch_kv_rms_norm_rope_cache(const KvLaunch& L, cudaStream_t stream);

}  // namespace ra
