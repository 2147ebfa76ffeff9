// C-ABI entry points of librope_attention.so (declared in include/rope_attention.h).
// Host-side validation happens here, before anything is launched.
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <string>

#include "rope_attention.h"
#include "internal.h"
#include "kv_cache.h"
#include "row_quant.h"

namespace ra {

int device_sm_count() {
  static std::atomic<int> cached{0};
  int v = cached.load();
  if (v > 0) return v;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  cached.store(n);
  return n;
}

}  // namespace ra

namespace {

thread_local std::string g_last_error;
std::atomic<int64_t> g_wait_ns{2000000000LL};
std::atomic<int> g_stall_next{0};  // ra_test_stall_next_projection
std::atomic<int> g_stall_next_kv{0};  // ra_test_stall_next_kv_cache
std::atomic<int> g_stall_next_norm{0};  // ra_test_stall_next_norm_rope
std::atomic<int> g_validate_only{0};    // ra_test_validate_only

// ra_test_validate_only: a call that passed its host checks returns here, before
// any CUDA runtime call
bool validate_only() { return g_validate_only.load() != 0; }

ra_status fail(ra_status code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
ra_status fail(ra_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

ra_status ok() {
  g_last_error.clear();
  return RA_OK;
}

ra_status cuda_fail(cudaError_t e, const char* where) {
  return fail(RA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct QkvShape {
  int64_t T, H, I;
  int32_t q_w, k_w;
  int32_t q_end, k_end;
  int32_t n_part_tiles;
  int32_t s_begin, s_end;   // Q/K columns carried as scaled fp16 between the passes
  int32_t ph_begin, ph_end; // Q/K columns finished in the projection (per-head norm)
  int32_t n_exp_blocks;     // 128-column blocks covering [0, s_end)
  int32_t part_stride, exp_stride;  // token-major row strides (16-byte multiples)
  size_t exps_offset;
  size_t workspace;
};

// which segments the norm/RoPE pass rewrites
// (across-heads norm, and RoPE whatever the norm: a per-head segment is normed in
// the projection and rotated here)
void second_pass_segments(const qkv_cte_mx_params* p, bool* do_q, bool* do_k) {
  *do_q = p->q_norm == RA_NORM_RMS_ACROSS_HEADS || p->fused_rope;
  *do_k = p->num_kv_heads > 0 && (p->k_norm == RA_NORM_RMS_ACROSS_HEADS || p->fused_rope);
}

ra_status check_params(const qkv_cte_mx_params* p, QkvShape* s) {
  if (p == nullptr) return fail(RA_ERR_INVALID_ARG, "params is NULL");
  if (p->B < 1 || p->S < 1) return fail(RA_ERR_INVALID_ARG, "B and S must be >= 1 (no empty tensors)");
  if (p->H < 128 || p->H % 128 != 0)
    return fail(RA_ERR_INVALID_ARG, "H must be a positive multiple of 128 (got %lld)",
                static_cast<long long>(p->H));
  if (p->num_heads < 1) return fail(RA_ERR_INVALID_ARG, "num_heads must be >= 1");
  if (p->num_kv_heads < 0) return fail(RA_ERR_INVALID_ARG, "num_kv_heads must be >= 0");
  if (p->head_dim < 16 || p->head_dim % 16 != 0)
    return fail(RA_ERR_INVALID_ARG, "head_dim must be a positive multiple of 16");
  if (p->q_norm != RA_NORM_NONE && p->q_norm != RA_NORM_RMS_ACROSS_HEADS && p->q_norm != RA_NORM_RMS_PER_HEAD)
    return fail(RA_ERR_INVALID_ARG, "q_norm must be an RA_NORM_* value");
  if (p->k_norm != RA_NORM_NONE && p->k_norm != RA_NORM_RMS_ACROSS_HEADS && p->k_norm != RA_NORM_RMS_PER_HEAD)
    return fail(RA_ERR_INVALID_ARG, "k_norm must be an RA_NORM_* value");
  if ((p->q_norm == RA_NORM_RMS_PER_HEAD || p->k_norm == RA_NORM_RMS_PER_HEAD) &&
      p->head_dim != 64 && p->head_dim != 128)
    return fail(RA_ERR_UNSUPPORTED, "the per-head norm is built for head_dim 64 and 128");
  if (p->k_norm != RA_NORM_NONE && p->num_kv_heads == 0)
    return fail(RA_ERR_INVALID_ARG, "k_norm needs a K segment (num_kv_heads == 0)");
  if (p->fused_rope != 0 && p->fused_rope != 1) return fail(RA_ERR_INVALID_ARG, "fused_rope must be 0 or 1");
  if (!(p->norm_eps >= 0.f) || !std::isfinite(p->norm_eps))
    return fail(RA_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
  if (p->output_layout != RA_LAYOUT_BSD && p->output_layout != RA_LAYOUT_NBSD)
    return fail(RA_ERR_INVALID_ARG, "unknown output_layout");
  const int64_t T = p->B * p->S;
  const int64_t I = static_cast<int64_t>(p->num_heads + 2 * p->num_kv_heads) * p->head_dim;
  if (T > 0x7fffffffLL || I > 0x7fffffffLL || p->H > 0x7fffffffLL || T * I > (1LL << 40))
    return fail(RA_ERR_INVALID_ARG, "problem too large for 32-bit tile coordinates");
  s->T = T;
  s->H = p->H;
  s->I = I;
  s->q_w = p->num_heads * p->head_dim;
  s->k_w = p->num_kv_heads * p->head_dim;
  s->q_end = s->q_w;
  s->k_end = s->q_w + s->k_w;
  const bool q_across = p->q_norm == RA_NORM_RMS_ACROSS_HEADS;
  const bool k_across = p->k_norm == RA_NORM_RMS_ACROSS_HEADS;
  const int32_t across_end = k_across ? s->k_end : (q_across ? s->q_end : 0);
  s->n_part_tiles = (q_across || k_across) ? (across_end + ra::kPartCols - 1) / ra::kPartCols : 0;
  // segments the second pass rewrites (across-heads norm, or RoPE without a norm) are
  // carried as scaled fp16 between the passes; per-head segments are finished in the
  // projection
  bool do_q, do_k;
  second_pass_segments(p, &do_q, &do_k);
  s->s_begin = do_q ? 0 : s->q_w;
  s->s_end = do_k ? s->k_end : s->q_w;
  if (!do_q && !do_k) s->s_begin = s->s_end = 0;
  const bool q_ph = p->q_norm == RA_NORM_RMS_PER_HEAD;
  const bool k_ph = p->num_kv_heads > 0 && p->k_norm == RA_NORM_RMS_PER_HEAD;
  s->ph_begin = q_ph ? 0 : s->q_w;
  s->ph_end = k_ph ? s->k_end : s->q_w;
  if (!q_ph && !k_ph) s->ph_begin = s->ph_end = 0;
  s->n_exp_blocks = (s->s_end + ra::kPartCols - 1) / ra::kPartCols;
  s->part_stride = (s->n_part_tiles + 1) / 2 * 2;
  s->exp_stride = (s->n_exp_blocks + 15) / 16 * 16;
  const size_t part = static_cast<size_t>(s->part_stride) * T * sizeof(float2);
  const size_t exps = static_cast<size_t>(s->exp_stride) * T;
  s->exps_offset = ra::kWorkspaceHeader + ((part + 255) / 256) * 256;
  s->workspace = s->exps_offset + ((exps + 255) / 256) * 256;
  return RA_OK;
}

ra_status check_project_inputs(const qkv_cte_mx_params* p, const uint8_t* a, const float* a_scale,
                               const void* w_packed, const float* ws, const uint16_t* bias,
                               const float* qg, const float* kg, const uint16_t* out) {
  if (!a || !a_scale || !w_packed || !out)
    return fail(RA_ERR_INVALID_ARG, "a, a_scale, w_packed and out are required");
  if (!aligned16(a) || !aligned16(out) || !aligned16(w_packed))
    return fail(RA_ERR_ALIGNMENT, "a, out and w_packed must be 16-byte aligned");
  if ((ws && !aligned16(ws)) || (bias && !aligned16(bias)))
    return fail(RA_ERR_ALIGNMENT, "weight_scales and bias must be 16-byte aligned");
  if (p->q_norm && !qg) return fail(RA_ERR_INVALID_ARG, "q_norm requires q_gamma");
  if (p->k_norm && !kg) return fail(RA_ERR_INVALID_ARG, "k_norm requires k_gamma");
  if ((qg && !aligned16(qg)) || (kg && !aligned16(kg)))
    return fail(RA_ERR_ALIGNMENT, "gammas must be 16-byte aligned");
  return RA_OK;
}

ra_status check_norm_inputs(const qkv_cte_mx_params* p, const float* cos, const float* sin,
                            const uint16_t* out) {
  if (!out) return fail(RA_ERR_INVALID_ARG, "out is required");
  if (!aligned16(out)) return fail(RA_ERR_ALIGNMENT, "out must be 16-byte aligned");
  if (p->fused_rope && (!cos || !sin))
    return fail(RA_ERR_INVALID_ARG, "fused_rope requires cos_cache and sin_cache");
  if ((cos && !aligned16(cos)) || (sin && !aligned16(sin)))
    return fail(RA_ERR_ALIGNMENT, "cos/sin caches must be 16-byte aligned");
  return RA_OK;
}

ra_status check_workspace(const void* workspace, size_t workspace_bytes, const QkvShape& s) {
  if (!workspace) return fail(RA_ERR_INVALID_ARG, "workspace is required");
  if (!aligned16(workspace)) return fail(RA_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  if (workspace_bytes < s.workspace)
    return fail(RA_ERR_WORKSPACE, "workspace too small: %zu < %zu", workspace_bytes, s.workspace);
  return RA_OK;
}

ra_status run_project(const qkv_cte_mx_params* p, const QkvShape& s, const uint8_t* a,
                      const float* a_scale, const void* w_packed, const float* ws,
                      const uint16_t* bias, const float* qg, const float* kg, uint16_t* out,
                      void* workspace, cudaStream_t st) {
  ra::ProjLaunch L{};
  L.a = a;
  L.a_scale = a_scale;
  L.w_t = static_cast<const uint8_t*>(w_packed);
  L.sf = static_cast<const uint8_t*>(w_packed) + ra::packed_sf_offset(s.H, s.I);
  L.weight_scales = ws;
  L.bias = bias;
  L.out = out;
  L.status = static_cast<int32_t*>(workspace);
  L.partials = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + ra::kWorkspaceHeader);
  L.T = s.T;
  L.H = s.H;
  L.I = s.I;
  L.q_end = s.q_end;
  L.k_end = p->num_kv_heads > 0 ? s.k_end : s.q_end;
  L.n_part_tiles = s.n_part_tiles;
  L.exps = reinterpret_cast<int8_t*>(static_cast<uint8_t*>(workspace) + s.exps_offset);
  L.n_exp_blocks = s.n_exp_blocks;
  L.part_stride = s.part_stride;
  L.exp_stride = s.exp_stride;
  L.s_begin = s.s_begin;
  L.s_end = s.s_end;
  // the gamma the epilogue folds in: across-heads segments only (the per-head
  // segments take theirs in the per-head norm)
  L.q_gamma = p->q_norm == RA_NORM_RMS_ACROSS_HEADS ? qg : nullptr;
  L.k_gamma = p->k_norm == RA_NORM_RMS_ACROSS_HEADS ? kg : nullptr;
  L.ph_begin = s.ph_begin;
  L.ph_end = s.ph_end;
  L.ph_q_gamma = p->q_norm == RA_NORM_RMS_PER_HEAD ? qg : nullptr;
  L.ph_k_gamma = p->k_norm == RA_NORM_RMS_PER_HEAD ? kg : nullptr;
  L.ph_carry = p->fused_rope;
  L.eps = p->norm_eps;
  L.wait_ns = g_wait_ns.load();
  L.stall_loads = g_stall_next.exchange(0);
  L.head_dim = p->head_dim;
  L.nbsd = p->output_layout == RA_LAYOUT_NBSD;
  const char* why = "launch failed";
  cudaError_t e = ra::launch_qkv_project(L, st, &why);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "qkv projection: %s (%s)", why, cudaGetErrorString(e));
  return RA_OK;
}

ra_status run_norm_rope(const qkv_cte_mx_params* p, const QkvShape& s, const float* cos,
                        const float* sin, uint16_t* out, void* workspace, cudaStream_t st) {
  bool do_q, do_k;
  second_pass_segments(p, &do_q, &do_k);
  if (!do_q && !do_k) return RA_OK;
  ra::NormRopeLaunch L{};
  L.out = out;
  L.partials =
      reinterpret_cast<const float2*>(static_cast<const uint8_t*>(workspace) + ra::kWorkspaceHeader);
  L.cos = cos;
  L.sin = sin;
  L.T = s.T;
  L.I = s.I;
  L.head_dim = p->head_dim;
  L.num_q_heads = p->num_heads;
  L.num_k_heads = p->num_kv_heads;
  L.q_norm = p->q_norm == RA_NORM_RMS_ACROSS_HEADS;
  L.k_norm = p->k_norm == RA_NORM_RMS_ACROSS_HEADS;
  L.rope = p->fused_rope;
  L.do_q = do_q;
  L.do_k = do_k;
  L.n_part_tiles = s.n_part_tiles;
  L.exps = reinterpret_cast<const int8_t*>(static_cast<const uint8_t*>(workspace) + s.exps_offset);
  L.part_stride = s.part_stride;
  L.n_exp_blocks = s.n_exp_blocks;
  L.exp_stride = s.exp_stride;
  L.eps = p->norm_eps;
  L.nbsd = p->output_layout == RA_LAYOUT_NBSD;
  L.status = static_cast<int32_t*>(workspace);
  L.wait_ns = g_wait_ns.load();
  L.stall_loads = g_stall_next_norm.exchange(0);
  cudaError_t e = ra::launch_qk_norm_rope(L, st);
  if (e != cudaSuccess) return cuda_fail(e, "norm/rope launch");
  return RA_OK;
}

}  // namespace

namespace ra {
void set_last_error(int code, const char* where, const char* what) {
  fail(static_cast<ra_status>(code), "%s: %s", where, what);
}

ra_status qkv_cte_mx_on_library_workspace(const qkv_cte_mx_params* p, const uint8_t* a,
                                          const float* a_scale, const void* w_packed,
                                          const float* weight_scales, const uint16_t* bias,
                                          const float* cos_cache, const float* sin_cache,
                                          const float* q_gamma, const float* k_gamma, uint16_t* out,
                                          size_t capacity, ra_status (*get_workspace)(void**),
                                          void* stream) {
  QkvShape s;
  ra_status st = check_params(p, &s);
  if (st != RA_OK) return st;
  if (s.workspace > capacity)
    return fail(RA_ERR_WORKSPACE,
                "qkv_cte_mx_noalloc: this call needs %zu bytes of scratch; the static workspace holds %zu",
                s.workspace, capacity);
  st = check_project_inputs(p, a, a_scale, w_packed, weight_scales, bias, q_gamma, k_gamma, out);
  if (st == RA_OK) st = check_norm_inputs(p, cos_cache, sin_cache, out);
  if (st != RA_OK) return st;
  if (validate_only()) return ok();
  void* ws = nullptr;
  st = get_workspace(&ws);
  if (st != RA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // the only scratch that must start at zero is the status word: the partial sums
  // and the exponents are written by the projection before the second pass reads them
  const cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int32_t), cs);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the static workspace status word");
  st = run_project(p, s, a, a_scale, w_packed, weight_scales, bias, q_gamma, k_gamma, out, ws, cs);
  if (st != RA_OK) return st;
  st = run_norm_rope(p, s, cos_cache, sin_cache, out, ws, cs);
  return st == RA_OK ? ok() : st;
}
}  // namespace ra

extern "C" {

const char* ra_last_error(void) { return g_last_error.c_str(); }

int32_t ra_abi_version(void) { return 9; }

void ra_set_wait_timeout_ns(int64_t ns) { g_wait_ns.store(ns < 1000 ? 1000 : ns); }

void ra_test_stall_next_projection(void) { g_stall_next.store(1); }

void ra_test_stall_next_kv_cache(void) { g_stall_next_kv.store(1); }

void ra_test_stall_next_norm_rope(void) { g_stall_next_norm.store(1); }

void ra_test_validate_only(int32_t on) { g_validate_only.store(on != 0 ? 1 : 0); }

ra_status qkv_cte_mx_packed_weight_bytes(int64_t H, int64_t I, size_t* bytes) {
  if (!bytes) return fail(RA_ERR_INVALID_ARG, "bytes is NULL");
  if (H < 128 || H % 128 != 0) return fail(RA_ERR_INVALID_ARG, "H must be a positive multiple of 128");
  if (I < 16 || I % 16 != 0) return fail(RA_ERR_INVALID_ARG, "I must be a positive multiple of 16");
  *bytes = ra::packed_weight_bytes(H, I);
  return ok();
}

ra_status qkv_cte_mx_pack_weight(const uint8_t* w, const uint8_t* w_block_exp, int64_t H, int64_t I,
                                 void* packed, size_t packed_bytes, void* stream) {
  size_t need = 0;
  ra_status st = qkv_cte_mx_packed_weight_bytes(H, I, &need);
  if (st != RA_OK) return st;
  if (!w || !w_block_exp || !packed) return fail(RA_ERR_INVALID_ARG, "w, w_block_exp and packed are required");
  if (!aligned16(packed)) return fail(RA_ERR_ALIGNMENT, "packed must be 16-byte aligned");
  if (packed_bytes < need) return fail(RA_ERR_WORKSPACE, "packed buffer too small: %zu < %zu", packed_bytes, need);
  if (H > 0x7fffffffLL || I > 0x7fffffffLL) return fail(RA_ERR_INVALID_ARG, "H or I too large");
  if (validate_only()) return ok();
  cudaError_t e = ra::launch_pack_weight(w, w_block_exp, H, I, static_cast<uint8_t*>(packed),
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pack_weight launch");
  return ok();
}

ra_status qkv_cte_mx_workspace_bytes(const qkv_cte_mx_params* p, size_t* bytes) {
  if (!bytes) return fail(RA_ERR_INVALID_ARG, "bytes is NULL");
  QkvShape s;
  ra_status st = check_params(p, &s);
  if (st != RA_OK) return st;
  *bytes = s.workspace;
  return ok();
}

ra_status qkv_cte_mx_project(const qkv_cte_mx_params* p, const uint8_t* a, const float* a_scale,
                             const void* w_packed, const float* weight_scales, const uint16_t* bias,
                             const float* q_gamma, const float* k_gamma, uint16_t* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  QkvShape s;
  ra_status st = check_params(p, &s);
  if (st == RA_OK) st = check_project_inputs(p, a, a_scale, w_packed, weight_scales, bias, q_gamma, k_gamma, out);
  if (st == RA_OK) st = check_workspace(workspace, workspace_bytes, s);
  if (st != RA_OK) return st;
  if (validate_only()) return ok();
  st = run_project(p, s, a, a_scale, w_packed, weight_scales, bias, q_gamma,
                   k_gamma, out, workspace, static_cast<cudaStream_t>(stream));
  return st == RA_OK ? ok() : st;
}

ra_status qkv_cte_mx_norm_rope(const qkv_cte_mx_params* p, const float* cos_cache,
                               const float* sin_cache, uint16_t* out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  QkvShape s;
  ra_status st = check_params(p, &s);
  if (st == RA_OK) st = check_norm_inputs(p, cos_cache, sin_cache, out);
  if (st == RA_OK) st = check_workspace(workspace, workspace_bytes, s);
  if (st != RA_OK) return st;
  if (validate_only()) return ok();
  st = run_norm_rope(p, s, cos_cache, sin_cache, out, workspace, static_cast<cudaStream_t>(stream));
  return st == RA_OK ? ok() : st;
}

ra_status qkv_cte_mx(const qkv_cte_mx_params* p, const uint8_t* a, const float* a_scale,
                     const void* w_packed, const float* weight_scales, const uint16_t* bias,
                     const float* cos_cache, const float* sin_cache, const float* q_gamma,
                     const float* k_gamma, uint16_t* out, void* workspace, size_t workspace_bytes,
                     void* stream) {
  QkvShape s;
  ra_status st = check_params(p, &s);
  if (st == RA_OK) st = check_project_inputs(p, a, a_scale, w_packed, weight_scales, bias, q_gamma, k_gamma, out);
  if (st == RA_OK) st = check_norm_inputs(p, cos_cache, sin_cache, out);
  if (st == RA_OK) st = check_workspace(workspace, workspace_bytes, s);
  if (st != RA_OK) return st;
  if (validate_only()) return ok();
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  st = run_project(p, s, a, a_scale, w_packed, weight_scales, bias, q_gamma,
                   k_gamma, out, workspace, cs);
  if (st != RA_OK) return st;
  st = run_norm_rope(p, s, cos_cache, sin_cache, out, workspace, cs);
  return st == RA_OK ? ok() : st;
}

ra_status qkv_cte_mx_status(void* workspace, void* stream, int32_t* device_status) {
  if (!device_status) return fail(RA_ERR_INVALID_ARG, "device_status is required");
  if (validate_only()) {
    *device_status = 0;
    return ok();
  }
  if (!workspace) {  // the static workspace of qkv_cte_mx_noalloc on the current device
    const ra_status st = ra::noalloc_workspace(&workspace);
    if (st != RA_OK) return st;
  }
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e == cudaSuccess && v != 0) e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *device_status = v;
  if (v != 0) return fail(RA_ERR_TIMEOUT, "a projection pipeline wait ran out of time (status %d)", v);
  return ok();
}

static ra_status row_quantize_common(const uint16_t* x, int64_t T, int64_t H, uint8_t* codes,
                                     float* scale, bool packed, void* stream) {
  if (!x || !codes || (!packed && !scale)) return fail(RA_ERR_INVALID_ARG, "x, codes (and scale) are required");
  if (T < 1 || H < 8 || H % 8 != 0 || H > (int64_t(1) << 30))
    return fail(RA_ERR_INVALID_ARG, "T >= 1 and H a positive multiple of 8 are required");
  if (!aligned16(x)) return fail(RA_ERR_ALIGNMENT, "x must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(codes) & (packed ? 3u : 7u)) != 0 ||
      (scale && (reinterpret_cast<uintptr_t>(scale) & 3u) != 0))
    return fail(RA_ERR_ALIGNMENT, packed ? "packed must be 4-byte aligned"
                                         : "codes must be 8-byte and scale 4-byte aligned");
  if (validate_only()) return ok();
  cudaError_t e = ra::launch_row_quantize(x, T, H, codes, scale, packed, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "row_quantize launch");
  return ok();
}

ra_status row_quantize_e4m3(const uint16_t* x, int64_t T, int64_t H, uint8_t* codes, float* scale,
                            void* stream) {
  return row_quantize_common(x, T, H, codes, scale, false, stream);
}

ra_status row_quantize_e4m3_packed(const uint16_t* x, int64_t T, int64_t H, uint8_t* packed,
                                   void* stream) {
  return row_quantize_common(x, T, H, packed, nullptr, true, stream);
}

ra_status kv_rms_norm_rope_cache(const kv_rms_norm_rope_cache_params* p, const uint16_t* kv,
                                 const uint16_t* gamma, const uint16_t* cos, const uint16_t* sin,
                                 const int64_t* index, void* k_cache, void* ckv_cache,
                                 const float* k_rope_scale, const float* c_kv_scale,
                                 const float* k_rope_offset, const float* c_kv_offset,
                                 const uint16_t* v_optional, uint16_t* k_rope, uint16_t* c_kv,
                                 int32_t* dev_error_count, void* stream) {
  if (p == nullptr) return fail(RA_ERR_INVALID_ARG, "params is NULL");
  if (!kv || !gamma || !cos || !sin || !index || !k_cache || !ckv_cache)
    return fail(RA_ERR_INVALID_ARG, "kv, gamma, cos, sin, index, k_cache and ckv_cache are required");
  if (p->B < 1 || p->N < 1 || p->S < 1 || p->Dkv < 1)
    return fail(RA_ERR_INVALID_ARG, "empty tensors are not supported");
  if (p->kv_dtype != RA_BF16 && p->kv_dtype != RA_FP16)
    return fail(RA_ERR_INVALID_ARG, "kv dtype must be bf16 or fp16");
  const int64_t R = p->rope_size;
  if (R < 8 || R % 8 != 0 || R > 256)
    return fail(RA_ERR_INVALID_ARG, "rope_size must be even; this build needs a multiple of 8 in [8, 256]");
  if (p->Dkv % 8 != 0 || p->Dv % 8 != 0 || p->Dv < 8)
    return fail(RA_ERR_INVALID_ARG, "Dkv and Dv must be positive multiples of 8");
  int64_t rms = 0;
  if (p->variant == 1) {
    if (p->N != 1) return fail(RA_ERR_INVALID_ARG, "V1 (combined kv) supports N == 1 only");
    if (v_optional) return fail(RA_ERR_INVALID_ARG, "v_optional must be NULL in V1");
    if (p->Dv != p->Dkv - R) return fail(RA_ERR_INVALID_ARG, "V1 needs Dv == Dkv - rope_size");
    rms = p->Dv;
  } else if (p->variant == 2) {
    if (!(p->N == 1 || p->N == 2 || p->N == 4 || p->N == 8))
      return fail(RA_ERR_INVALID_ARG, "V2 (separate kv) supports N in {1, 2, 4, 8}");
    if (!v_optional) return fail(RA_ERR_INVALID_ARG, "V2 needs v_optional");
    if (R > p->Dkv) return fail(RA_ERR_INVALID_ARG, "rope_size exceeds Dkv");
    if (p->Dv > 1024) return fail(RA_ERR_INVALID_ARG, "V2 needs Dv <= 1024 in this build");
    rms = p->Dkv;
  } else {
    return fail(RA_ERR_INVALID_ARG, "variant must be 1 or 2");
  }
  if (rms < 8 || rms > 1024) return fail(RA_ERR_INVALID_ARG, "rms_size must be in [8, 1024]");
  if ((k_rope_offset && !k_rope_scale) || (c_kv_offset && !c_kv_scale))
    return fail(RA_ERR_INVALID_ARG, "an offset without its scale is illegal");
  const bool qk = k_rope_scale != nullptr, qv = c_kv_scale != nullptr;
  auto quant_type = [](int32_t d) -> int32_t {
    return d == RA_INT8 ? ra::kQuantInt8 : d == RA_FP8_E4M3 ? ra::kQuantE4m3 : d == RA_FP8_E5M2 ? ra::kQuantE5m2 : -1;
  };
  const int32_t kq = qk ? quant_type(p->k_cache_dtype) : 0;
  const int32_t vq = qv ? quant_type(p->ckv_cache_dtype) : 0;
  if (qk ? kq < 0 : p->k_cache_dtype != p->kv_dtype)
    return fail(RA_ERR_INVALID_ARG, "k_cache dtype must be int8 or fp8 with a k scale, else equal to the kv dtype");
  if (qv ? vq < 0 : p->ckv_cache_dtype != p->kv_dtype)
    return fail(RA_ERR_INVALID_ARG, "ckv_cache dtype must be int8 or fp8 with a c_kv scale, else equal to the kv dtype");
  const int32_t mode = p->cache_mode;
  if (mode == RA_CACHE_PA_NZ || mode == RA_CACHE_PA_BLK_NZ)
    return fail(RA_ERR_UNSUPPORTED, "FRACTAL_NZ cache modes are not built");
  if (mode != RA_CACHE_NORM && mode != RA_CACHE_PA && mode != RA_CACHE_PA_BNSD && mode != RA_CACHE_PA_BLK_BNSD)
    return fail(RA_ERR_INVALID_ARG, "unknown cache_mode");
  if (mode == RA_CACHE_NORM) {
    if (p->cache_seq_len < p->S) return fail(RA_ERR_INVALID_ARG, "NORM mode needs cache_seq_len >= S");
    if (p->variant == 1 && (qk || qv))
      return fail(RA_ERR_INVALID_ARG, "V1 in NORM mode takes no quantisation parameters");
  } else {
    if (p->block_num < 1 || p->block_size <= 1)
      return fail(RA_ERR_INVALID_ARG, "block_num >= 1 and block_size > 1 are required");
    if ((qk || qv) && p->block_size % 32 != 0)
      return fail(RA_ERR_INVALID_ARG, "1-byte caches need block_size %% 32 == 0");
    if ((!qk || !qv) && p->block_size % 16 != 0)
      return fail(RA_ERR_INVALID_ARG, "2-byte caches need block_size %% 16 == 0");
  }
  if ((p->k_quant_scalar != 0 && p->k_quant_scalar != 1) || (p->c_kv_quant_scalar != 0 && p->c_kv_quant_scalar != 1))
    return fail(RA_ERR_INVALID_ARG, "k_quant_scalar and c_kv_quant_scalar must be 0 or 1");
  if (p->variant == 2 && (p->k_quant_scalar || p->c_kv_quant_scalar))
    return fail(RA_ERR_INVALID_ARG, "V2 quantisation parameters are [N, D]; the [1] form is V1 only");
  if ((p->k_quant_scalar && !qk) || (p->c_kv_quant_scalar && !qv))
    return fail(RA_ERR_INVALID_ARG, "a [1] quantisation parameter flag needs its scale");
  if (p->rope_s_broadcast != 0 && p->rope_s_broadcast != 1)
    return fail(RA_ERR_INVALID_ARG, "rope_s_broadcast must be 0 or 1");
  if (!(p->epsilon >= 0.f) || !std::isfinite(p->epsilon))
    return fail(RA_ERR_INVALID_ARG, "epsilon must be finite and >= 0");
  const bool outputs = p->is_output_kv && (mode != RA_CACHE_NORM || (p->variant == 2 && (qk || qv)));
  if (outputs && (!k_rope || !c_kv))
    return fail(RA_ERR_INVALID_ARG, "is_output_kv requires k_rope and c_kv");
  if (!aligned16(kv) || !aligned16(gamma) || !aligned16(cos) || !aligned16(sin) ||
      !aligned16(k_cache) || !aligned16(ckv_cache) || (v_optional && !aligned16(v_optional)) ||
      (k_rope && !aligned16(k_rope)) || (c_kv && !aligned16(c_kv)) ||
      (k_rope_scale && !aligned16(k_rope_scale)) || (c_kv_scale && !aligned16(c_kv_scale)) ||
      (k_rope_offset && !aligned16(k_rope_offset)) || (c_kv_offset && !aligned16(c_kv_offset)) ||
      (reinterpret_cast<uintptr_t>(index) & 7u))
    return fail(RA_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned (index 8-byte)");
  if (p->B * p->N * p->S > (1LL << 40)) return fail(RA_ERR_INVALID_ARG, "too many rows");
  if (mode == RA_CACHE_NORM && p->cache_seq_len > (1LL << 31)) return fail(RA_ERR_INVALID_ARG, "cache_seq_len too large");
  if (p->S > (1LL << 31)) return fail(RA_ERR_INVALID_ARG, "S too large");
  if (validate_only()) return ok();

  ra::KvLaunch L{};
  L.kv = kv;
  L.gamma = gamma;
  L.cos = cos;
  L.sin = sin;
  L.index = index;
  L.k_cache = k_cache;
  L.ckv_cache = ckv_cache;
  L.k_scale = k_rope_scale;
  L.k_offset = k_rope_offset;
  L.v_scale = c_kv_scale;
  L.v_offset = c_kv_offset;
  L.v = v_optional;
  L.k_rope = k_rope;
  L.c_kv = c_kv;
  L.err_count = dev_error_count;
  L.B = p->B;
  L.N = p->N;
  L.S = p->S;
  L.Dkv = p->Dkv;
  L.Dv = p->Dv;
  L.R = p->rope_size;
  L.variant = p->variant;
  L.mode = p->cache_mode;
  L.block_num = p->block_num;
  L.block_size = p->block_size;
  L.eps = p->epsilon;
  L.out_kv = outputs;
  L.f16 = p->kv_dtype == RA_FP16;
  L.kq = kq;
  L.vq = vq;
  L.rope_bcast = p->rope_s_broadcast;
  L.k_scalar = p->k_quant_scalar;
  L.v_scalar = p->c_kv_quant_scalar;
  L.cache_seq = mode == RA_CACHE_NORM ? p->cache_seq_len : 0;
  L.wait_ns = g_wait_ns.load();
  L.stall_loads = g_stall_next_kv.exchange(0);
  L.status = ra::kv_status_word();
  cudaError_t e = ra::launch_kv_rms_norm_rope_cache(L, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_rms_norm_rope_cache launch");
  return ok();
}

ra_status kv_rms_norm_rope_cache_status(void* stream, int32_t* device_status) {
  if (!device_status) return fail(RA_ERR_INVALID_ARG, "device_status is required");
  if (validate_only()) {
    *device_status = 0;
    return ok();
  }
  int32_t* word = ra::kv_status_word();
  if (!word) return fail(RA_ERR_CUDA, "the KV status word cannot be found on this device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v != 0) e = cudaMemsetAsync(word, 0, sizeof(v), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "KV status read");
  *device_status = v;
  if (v != 0) return fail(RA_ERR_TIMEOUT, "a KV cache pipeline wait ran out of time (status %d)", v);
  return ok();
}

}  // extern "C"
