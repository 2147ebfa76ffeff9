/* Example: the attention prologue of one Wan2.2-style self-attention layer from
 * C, with the CUDA runtime for memory.  Compiled (not run) by
 * tests/test_c_abi.py; it needs a GPU to run.
 *
 *   setup:    pack W once, size and zero the workspace once
 *   per step: qkv_cte_mx on the layer's activations, then the KV-cache update;
 *             read the device status words when convenient (they synchronise). */
#include <stdio.h>

#include <cuda_runtime_api.h>

#include "rope_attention.h"

#define CHECK_RA(call)                                                        \
  do {                                                                        \
    ra_status s_ = (call);                                                    \
    if (s_ != RA_OK) {                                                        \
      fprintf(stderr, "%s failed (%d): %s\n", #call, (int)s_, ra_last_error()); \
      return -1;                                                              \
    }                                                                         \
  } while (0)

typedef struct {
  qkv_cte_mx_params p;
  void* w_packed;  /* qkv_cte_mx_packed_weight_bytes(H, I) */
  void* workspace; /* qkv_cte_mx_workspace_bytes(&p)        */
  size_t workspace_bytes;
} prologue;

/* w [H, I] E4M3 codes and w_block_exp [H/32, I] UE8M0 exponents, on the device. */
int prologue_setup(prologue* pr, int64_t S, const uint8_t* w, const uint8_t* w_block_exp,
                   cudaStream_t stream) {
  size_t packed_bytes = 0;
  qkv_cte_mx_params* p = &pr->p;
  p->B = 1;
  p->S = S;
  p->H = 5120;
  p->num_heads = 40;
  p->num_kv_heads = 40;
  p->head_dim = 128;
  p->q_norm = RA_NORM_RMS_ACROSS_HEADS;
  p->k_norm = RA_NORM_RMS_ACROSS_HEADS;
  p->fused_rope = 1;
  p->norm_eps = 1e-6f;
  p->output_layout = RA_LAYOUT_BSD;
  {
    const int64_t I = (int64_t)(p->num_heads + 2 * p->num_kv_heads) * p->head_dim;
    CHECK_RA(qkv_cte_mx_packed_weight_bytes(p->H, I, &packed_bytes));
    if (cudaMalloc(&pr->w_packed, packed_bytes) != cudaSuccess) return -1;
    CHECK_RA(qkv_cte_mx_pack_weight(w, w_block_exp, p->H, I, pr->w_packed, packed_bytes, stream));
  }
  CHECK_RA(qkv_cte_mx_workspace_bytes(p, &pr->workspace_bytes));
  if (cudaMalloc(&pr->workspace, pr->workspace_bytes) != cudaSuccess) return -1;
  if (cudaMemsetAsync(pr->workspace, 0, pr->workspace_bytes, stream) != cudaSuccess) return -1;
  return 0;
}

/* One step.  a [S, H] E4M3 codes and a_scale [S] from row_quantize_e4m3; cos/sin
 * [S, 128] fp32 rotate-half tables; gammas [5120] fp32; bias [15360] bf16 bits;
 * out [S, 15360] bf16 bits.  kv / v / caches as in the header's
 * kv_rms_norm_rope_cache comment, with kvp describing them. */
int prologue_step(prologue* pr, const uint16_t* hidden, uint8_t* a, float* a_scale, const uint16_t* bias,
                  const float* cos_cache, const float* sin_cache, const float* q_gamma, const float* k_gamma,
                  uint16_t* out, const kv_rms_norm_rope_cache_params* kvp, const uint16_t* kv,
                  const uint16_t* kv_gamma, const uint16_t* kv_cos, const uint16_t* kv_sin, const int64_t* index,
                  void* k_cache, void* ckv_cache, const float* k_scale, const float* v_scale,
                  const float* k_offset, const float* v_offset, const uint16_t* v, cudaStream_t stream) {
  CHECK_RA(row_quantize_e4m3(hidden, pr->p.B * pr->p.S, pr->p.H, a, a_scale, stream));
  CHECK_RA(qkv_cte_mx(&pr->p, a, a_scale, pr->w_packed, NULL, bias, cos_cache, sin_cache, q_gamma, k_gamma,
                      out, pr->workspace, pr->workspace_bytes, stream));
  CHECK_RA(kv_rms_norm_rope_cache(kvp, kv, kv_gamma, kv_cos, kv_sin, index, k_cache, ckv_cache, k_scale, v_scale,
                                  k_offset, v_offset, v, NULL, NULL, NULL, stream));
  return 0;
}

/* After a synchronisation point: did any device pipeline wait give up? */
int prologue_check(prologue* pr, cudaStream_t stream) {
  int32_t qkv_word = 0, kv_word = 0;
  CHECK_RA(qkv_cte_mx_status(pr->workspace, stream, &qkv_word));
  CHECK_RA(kv_rms_norm_rope_cache_status(stream, &kv_word));
  return qkv_word == 0 && kv_word == 0 ? 0 : -1;
}
