/* The attention prologue run from C on a GPU, for tests/test_c_abi_gpu.py.
 *
 * Reads a seeded problem from raw little-endian files in DIR (written by the
 * test), allocates device memory with the CUDA runtime, and makes the calls a C
 * user of the library makes: the row quantiser on the bf16 hidden state, the
 * one-time weight packing, qkv_cte_mx, kv_rms_norm_rope_cache and the two status
 * readers.  Writes the results back to DIR for the test to compare with the
 * oracle.
 *
 *   prologue_gpu DIR S H NQ NKV D  B N SKV DKV DV BS BN
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "rope_attention.h"

static char g_dir[1024];

static int fail(const char* what, const char* why) {
  fprintf(stderr, "%s: %s\n", what, why);
  return 1;
}

static void* read_file(const char* name, size_t bytes) {
  char path[1200];
  FILE* f;
  void* buf = malloc(bytes ? bytes : 1);
  snprintf(path, sizeof path, "%s/%s", g_dir, name);
  f = fopen(path, "rb");
  if (!f || !buf || fread(buf, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot read %zu bytes of %s\n", bytes, path);
    exit(2);
  }
  fclose(f);
  return buf;
}

static void write_file(const char* name, const void* buf, size_t bytes) {
  char path[1200];
  FILE* f;
  snprintf(path, sizeof path, "%s/%s", g_dir, name);
  f = fopen(path, "wb");
  if (!f || fwrite(buf, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot write %s\n", path);
    exit(2);
  }
  fclose(f);
}

/* a device copy of a host file */
static void* to_device(const char* name, size_t bytes) {
  void* h = read_file(name, bytes);
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess || cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
    fprintf(stderr, "device copy of %s failed\n", name);
    exit(2);
  }
  free(h);
  return d;
}

static void from_device(const char* name, const void* d, size_t bytes) {
  void* h = malloc(bytes);
  if (!h || cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
    fprintf(stderr, "device read of %s failed\n", name);
    exit(2);
  }
  write_file(name, h, bytes);
  free(h);
}

#define CHECK_RA(call)                                                \
  do {                                                                \
    ra_status s_ = (call);                                            \
    if (s_ != RA_OK) return fail(#call, ra_last_error());             \
  } while (0)

int main(int argc, char** argv) {
  qkv_cte_mx_params q;
  kv_rms_norm_rope_cache_params kv;
  int64_t S, H, T, I, B, N, SKV, DKV, DV, BS, BN, rows;
  int nq, nkv, d;
  size_t packed_bytes = 0, ws_bytes = 0;
  void *hidden, *w, *w_exp, *bias, *cos_q, *sin_q, *qg, *kg, *a, *a_scale, *packed, *ws, *out;
  void *kvx, *gamma, *cos_k, *sin_k, *index, *kc, *cc, *ks, *ko, *vs, *vo, *v, *err;
  int32_t word = 0;
  cudaStream_t st;

  if (argc != 14) return fail("usage", "prologue_gpu DIR S H NQ NKV D B N SKV DKV DV BS BN");
  snprintf(g_dir, sizeof g_dir, "%s", argv[1]);
  S = atoll(argv[2]); H = atoll(argv[3]); nq = atoi(argv[4]); nkv = atoi(argv[5]); d = atoi(argv[6]);
  B = atoll(argv[7]); N = atoll(argv[8]); SKV = atoll(argv[9]); DKV = atoll(argv[10]); DV = atoll(argv[11]);
  BS = atoll(argv[12]); BN = atoll(argv[13]);
  T = S;
  I = (int64_t)(nq + 2 * nkv) * d;
  rows = B * N * SKV;
  if (cudaStreamCreate(&st) != cudaSuccess) return fail("cudaStreamCreate", "failed");

  /* (a) the projection prologue: quantise, pack, project, norm + RoPE */
  hidden = to_device("hidden.bin", (size_t)(T * H * 2));
  w = to_device("w.bin", (size_t)(H * I));
  w_exp = to_device("w_exp.bin", (size_t)(H / 32 * I));
  bias = to_device("bias.bin", (size_t)(I * 2));
  cos_q = to_device("cos_q.bin", (size_t)(T * d * 4));
  sin_q = to_device("sin_q.bin", (size_t)(T * d * 4));
  qg = to_device("q_gamma.bin", (size_t)nq * d * 4);
  kg = to_device("k_gamma.bin", (size_t)nkv * d * 4);
  if (cudaMalloc(&a, (size_t)(T * H)) != cudaSuccess || cudaMalloc(&a_scale, (size_t)(T * 4)) != cudaSuccess ||
      cudaMalloc(&out, (size_t)(T * I * 2)) != cudaSuccess)
    return fail("cudaMalloc", "activation / output");

  memset(&q, 0, sizeof q);
  q.B = 1;
  q.S = S;
  q.H = H;
  q.num_heads = nq;
  q.num_kv_heads = nkv;
  q.head_dim = d;
  q.q_norm = RA_NORM_RMS_ACROSS_HEADS;
  q.k_norm = RA_NORM_RMS_ACROSS_HEADS;
  q.fused_rope = 1;
  q.norm_eps = 1e-6f;
  q.output_layout = RA_LAYOUT_BSD;
  CHECK_RA(qkv_cte_mx_packed_weight_bytes(H, I, &packed_bytes));
  if (cudaMalloc(&packed, packed_bytes) != cudaSuccess) return fail("cudaMalloc", "packed weight");
  CHECK_RA(qkv_cte_mx_pack_weight((const uint8_t*)w, (const uint8_t*)w_exp, H, I, packed, packed_bytes, st));
  CHECK_RA(qkv_cte_mx_workspace_bytes(&q, &ws_bytes));
  if (cudaMalloc(&ws, ws_bytes) != cudaSuccess || cudaMemsetAsync(ws, 0, ws_bytes, st) != cudaSuccess)
    return fail("cudaMalloc", "workspace");
  CHECK_RA(row_quantize_e4m3((const uint16_t*)hidden, T, H, (uint8_t*)a, (float*)a_scale, st));
  CHECK_RA(qkv_cte_mx(&q, (const uint8_t*)a, (const float*)a_scale, packed, NULL, (const uint16_t*)bias,
                      (const float*)cos_q, (const float*)sin_q, (const float*)qg, (const float*)kg,
                      (uint16_t*)out, ws, ws_bytes, st));

  /* (b) the KV-cache update: V2, int8 per-head quantisation, PA_BNSD */
  kvx = to_device("kv.bin", (size_t)(rows * DKV * 2));
  v = to_device("v.bin", (size_t)(rows * DV * 2));
  gamma = to_device("kv_gamma.bin", (size_t)(DKV * 2));
  cos_k = to_device("cos_k.bin", (size_t)(rows * 64 * 2));
  sin_k = to_device("sin_k.bin", (size_t)(rows * 64 * 2));
  index = to_device("index.bin", (size_t)(B * SKV * 8));
  kc = to_device("k_cache.bin", (size_t)(BN * N * BS * DKV));
  cc = to_device("ckv_cache.bin", (size_t)(BN * N * BS * DV));
  ks = to_device("k_scale.bin", (size_t)(N * DKV * 4));
  ko = to_device("k_offset.bin", (size_t)(N * DKV * 4));
  vs = to_device("v_scale.bin", (size_t)(N * DV * 4));
  vo = to_device("v_offset.bin", (size_t)(N * DV * 4));
  if (cudaMalloc(&err, 4) != cudaSuccess || cudaMemset(err, 0, 4) != cudaSuccess)
    return fail("cudaMalloc", "error counter");
  memset(&kv, 0, sizeof kv);
  kv.B = B;
  kv.N = N;
  kv.S = SKV;
  kv.Dkv = DKV;
  kv.Dv = DV;
  kv.rope_size = 64;
  kv.variant = 2;
  kv.cache_mode = RA_CACHE_PA_BNSD;
  kv.block_num = BN;
  kv.block_size = BS;
  kv.kv_dtype = RA_BF16;
  kv.k_cache_dtype = RA_INT8;
  kv.ckv_cache_dtype = RA_INT8;
  kv.epsilon = 1e-5f;
  kv.is_output_kv = 0;
  CHECK_RA(kv_rms_norm_rope_cache(&kv, (const uint16_t*)kvx, (const uint16_t*)gamma, (const uint16_t*)cos_k,
                                  (const uint16_t*)sin_k, (const int64_t*)index, kc, cc, (const float*)ks,
                                  (const float*)vs, (const float*)ko, (const float*)vo, (const uint16_t*)v, NULL,
                                  NULL, (int32_t*)err, st));

  /* status words (these synchronise the stream) */
  CHECK_RA(qkv_cte_mx_status(ws, st, &word));
  if (word != 0) return fail("qkv_cte_mx_status", "a pipeline wait ran out");
  CHECK_RA(kv_rms_norm_rope_cache_status(st, &word));
  if (word != 0) return fail("kv_rms_norm_rope_cache_status", "a pipeline wait ran out");

  from_device("a_out.bin", a, (size_t)(T * H));
  from_device("a_scale_out.bin", a_scale, (size_t)(T * 4));
  from_device("out.bin", out, (size_t)(T * I * 2));
  from_device("k_cache_out.bin", kc, (size_t)(BN * N * BS * DKV));
  from_device("ckv_cache_out.bin", cc, (size_t)(BN * N * BS * DV));
  from_device("err_out.bin", err, 4);
  printf("prologue ok\n");
  return 0;
}
