/* A C99 caller of librope_attention.so: includes the public header, links
 * against the library and makes the calls that need no GPU (version, size
 * queries, host-side validation).  Prints one "name value" line per result
 * for tests/test_c_abi.py to compare with the Python binding. */
#include <stdio.h>
#include <string.h>

#include "rope_attention.h"

int main(void) {
  qkv_cte_mx_params q;
  kv_rms_norm_rope_cache_params kv;
  size_t bytes = 0;
  ra_status st;

  /* the calls below hand the library placeholder addresses: with this hook set a
   * call that passed its checks would return before touching CUDA */
  ra_test_validate_only(1);
  printf("abi %d\n", (int)ra_abi_version());

  st = qkv_cte_mx_packed_weight_bytes(5120, 15360, &bytes);
  printf("packed_status %d\npacked_bytes %zu\n", (int)st, bytes);

  /* the 720p self-attention call: 40 + 40 + 40 heads of 128, across-heads norms, RoPE */
  memset(&q, 0, sizeof q);
  q.B = 1;
  q.S = 75600;
  q.H = 5120;
  q.num_heads = 40;
  q.num_kv_heads = 40;
  q.head_dim = 128;
  q.q_norm = RA_NORM_RMS_ACROSS_HEADS;
  q.k_norm = RA_NORM_RMS_ACROSS_HEADS;
  q.fused_rope = 1;
  q.norm_eps = 1e-6f;
  q.output_layout = RA_LAYOUT_BSD;
  st = qkv_cte_mx_workspace_bytes(&q, &bytes);
  printf("workspace_status %d\nworkspace_bytes %zu\n", (int)st, bytes);

  /* rejected on the host: H not a multiple of 128 */
  q.H = 5000;
  st = qkv_cte_mx_workspace_bytes(&q, &bytes);
  printf("bad_h_status %d\nbad_h_message %s\n", (int)st, ra_last_error());

  /* rejected on the host before any pointer is used: V1 with N != 1 */
  memset(&kv, 0, sizeof kv);
  kv.B = 1;
  kv.N = 2;
  kv.S = 4;
  kv.Dkv = 576;
  kv.Dv = 512;
  kv.rope_size = 64;
  kv.variant = 1;
  kv.cache_mode = RA_CACHE_PA_BNSD;
  kv.block_num = 1;
  kv.block_size = 16;
  kv.kv_dtype = RA_BF16;
  kv.k_cache_dtype = RA_BF16;
  kv.ckv_cache_dtype = RA_BF16;
  kv.epsilon = 1e-5f;
  {
    static uint16_t placeholder[8];
    int64_t index[1] = {0};
    st = kv_rms_norm_rope_cache(&kv, placeholder, placeholder, placeholder, placeholder, index, placeholder,
                                placeholder, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL);
  }
  printf("kv_v1_n2_status %d\nkv_v1_n2_message %s\n", (int)st, ra_last_error());
  return 0;
}
