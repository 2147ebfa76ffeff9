// Internal interfaces between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <mutex>

#include "rope_attention.h"

namespace ra {

// ------------------------------------------------------------ projection (K1)
// Tile shape of the block-scaled FP8 GEMM; also fixes the packed weight layout.
constexpr int kProjBN = 256;          // output columns per CTA-pair tile (256 rows x 256 columns)
constexpr int kProjBK = 128;          // contraction elements (= bytes) per pipeline stage
constexpr int kPartCols = 128;        // columns covered by one sum-of-squares partial
// W's block scales of one (256-column pair tile, 128-deep K stage): a 4 KB image of
// 128 rows x 32 bytes (TMEM lane L: the 4 block scales of columns c * 32 + L % 32,
// c = 0..7), copied into TMEM by one tcgen05.cp 128x256b
constexpr int kSfStageBytes = 4096;
constexpr int kWorkspaceHeader = 256; // status word + padding, ahead of the partial sums

struct ProjLaunch {
  const uint8_t* a;            // [T, H] e4m3
  const float* a_scale;        // [T]
  const uint8_t* w_t;          // [I, H] e4m3 (packed, K-major)
  const uint8_t* sf;           // packed block-scale images (4 KB per column tile and K stage)
  const float* weight_scales;  // [I] or null
  const uint16_t* bias;        // [I] bf16 or null
  uint16_t* out;               // [T, I]: bf16, except columns [s_begin, s_end) (see below)
  int8_t* exps;                // [T, exp_stride] power-of-two exponent per 128-column block
  float2* partials;            // [T, part_stride] (sum sq Q, sum sq K) per 128-column block
  int32_t* status;
  int64_t T, H, I;
  int32_t q_end, k_end;        // Q = [0, q_end), K = [q_end, k_end) output columns
  int32_t s_begin, s_end;      // Q/K columns the second pass rewrites: stored as fp16 of
                               // z * 2^-e, e per (row, 128-column block) in `exps`, with
                               // z = v * gamma
  int32_t n_part_tiles, part_stride;   // part_stride = n_part_tiles rounded up to even
  int32_t n_exp_blocks, exp_stride;    // exp_stride = n_exp_blocks rounded up to 16
  // applied before the encoding (it commutes with inv_rms and the rotation):
  const float* q_gamma;        // [q_end] gamma of a normed Q segment, or null
  const float* k_gamma;        // [k_end - q_end] gamma of a normed K segment, or null
  int64_t wait_ns;
  int32_t stall_loads;         // test hook: issue no TMA loads, so the pipeline waits run out
  int32_t head_dim;
  int32_t nbsd;                // out is [I / head_dim, T, head_dim] instead of [T, I]
  // columns [ph_begin, ph_end) take the per-head norm in the epilogue: finished
  // there (bf16) without RoPE, or normed and carried to the RoPE pass (ph_carry)
  int32_t ph_begin, ph_end;
  const float* ph_q_gamma;     // [head_dim] per-head gamma of the Q / K segment, or null
  const float* ph_k_gamma;
  int32_t ph_carry;
  float eps;
};
cudaError_t launch_qkv_project(const ProjLaunch& L, cudaStream_t stream, const char** why);

size_t packed_weight_bytes(int64_t H, int64_t I);
size_t packed_sf_offset(int64_t H, int64_t I);
cudaError_t launch_pack_weight(const uint8_t* w, const uint8_t* w_block_exp, int64_t H, int64_t I,
                               uint8_t* packed, cudaStream_t stream);

// ------------------------------------------------------------ norm + RoPE apply (K2)
struct NormRopeLaunch {
  uint16_t* out;               // [T, I]: encoded Q/K in, bf16 normed / rotated Q/K out
  const int8_t* exps;          // [T, exp_stride] exponents of the scaled fp16 encoding
  const float2* partials;      // [T, part_stride]
  const float* cos;            // [T, d], used when rope
  const float* sin;
  int64_t T, I;
  int32_t head_dim, num_q_heads, num_k_heads;
  int32_t q_norm, k_norm, rope;
  int32_t n_part_tiles, part_stride;
  int32_t n_exp_blocks, exp_stride;
  float eps;
  int32_t nbsd;                // out is [I / head_dim, T, head_dim] instead of [T, I]
  int32_t do_q, do_k;          // segments this pass rewrites
  int32_t* status;             // workspace status word (pipelined kernel: a wait ran out)
  int64_t wait_ns;             // time limit of each pipeline wait
  int32_t stall_loads;         // test hook: the pipelined kernel issues no copies
};
cudaError_t launch_qk_norm_rope(const NormRopeLaunch& L, cudaStream_t stream);

int device_sm_count();

// cuTensorMapEncodeTiled, looked up once through the runtime (null if unavailable)
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Sets the thread-local message returned by ra_last_error() ("where: what").
void set_last_error(int code, const char* where, const char* what);

// ------------------------------------------------------------ qkv_cte_mx_noalloc
// The whole qkv_cte_mx call on a workspace the library owns: every host check of
// qkv_cte_mx (and the problem's scratch against `capacity`) first; then
// `get_workspace` supplies the workspace's device address, its status word is
// cleared on `stream` and both passes launch.  Nothing is enqueued for a rejected call.
ra_status qkv_cte_mx_on_library_workspace(const qkv_cte_mx_params* p, const uint8_t* a,
                                          const float* a_scale, const void* w_packed,
                                          const float* weight_scales, const uint16_t* bias,
                                          const float* cos_cache, const float* sin_cache,
                                          const float* q_gamma, const float* k_gamma, uint16_t* out,
                                          size_t capacity, ra_status (*get_workspace)(void**),
                                          void* stream);
// Device address of qkv_cte_mx_noalloc's static workspace on the current device
// (looked up once per device).
ra_status noalloc_workspace(void** ws);

}  // namespace ra
