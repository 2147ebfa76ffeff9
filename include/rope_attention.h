/*
 * rope_attention.h -- C ABI of librope_attention.so, the GB300 (sm_103a)
 * attention-prologue hot path.
 *
 * Two operators:
 *
 *  (a) qkv_cte_mx: the fused QKV projection of the AWS Neuron page "Kernel
 *      reference: qkv_cte -- Wan2.2 additions to the NKI Library QKV CTE MXFP8
 *      projection" (sections "Applies to"/Pattern, "Upstream behavior",
 *      Design 1 across-heads RMSNorm, Design 2 rotate-half RoPE, Design 5
 *      single-segment calls, "Interface"):
 *        O[T, I] = dequant(A[T, H]) @ dequant(W[H, I]) + bias,
 *        I = (num_heads + 2*num_kv_heads) * head_dim, T = B*S,
 *      then, per token, one RMS over the whole Q segment and one over the
 *      whole K segment, the segment-wide gamma, and rotate-half RoPE on Q and
 *      K, written back in place; V is left as projected.
 *
 *  (b) kv_rms_norm_rope_cache: the CANN ops-transformer operator
 *      "KvRmsNormRopeCache" (formulas (1) RmsNorm, (2) interleaveRope,
 *      (3) quantisation, (4) scatter, (5) is_output_kv; parameter table;
 *      cache/index constraint table), modes V1 (combined kv) and V2
 *      (separate kv with v_optional).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensor pointers are DEVICE pointers owned by the caller, dense and
 *    row-major (last dimension contiguous) unless stated otherwise.  The hot
 *    calls allocate nothing; scratch space is the caller's workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is asynchronous and stream-ordered; no call
 *    synchronises except the *_status readers.
 *  - Arguments are validated on the host before anything is launched; a
 *    rejected call returns a negative ra_status, launches nothing and sets
 *    the thread-local message returned by ra_last_error().  RA_ERR_CUDA
 *    means a CUDA runtime call failed (message carries cudaGetErrorString).
 *  - Device-side conditions (a pipeline wait that ran out of time, an index
 *    out of range) never trap: they are recorded in device memory that the
 *    caller reads after synchronising (qkv_cte_mx_status,
 *    kv_rms_norm_rope_cache_status, dev_error_count).
 *  - bf16 values are passed as their 16-bit patterns (uint16_t).
 *  - qkv_cte_mx, qkv_cte_mx_project, qkv_cte_mx_norm_rope, row_quantize_e4m3,
 *    row_quantize_e4m3_packed, qkv_cte_mx_pack_weight and kv_rms_norm_rope_cache
 *    launch kernels only (no allocation, no synchronisation), so after one
 *    eager call per device they can be captured into a CUDA graph and
 *    replayed; the status readers synchronise and cannot be captured.
 */
#ifndef ROPE_ATTENTION_H_
#define ROPE_ATTENTION_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = -1,   /* bad shape, null pointer, illegal combination          */
  RA_ERR_UNSUPPORTED = -2,   /* legal on the pages but not built here                  */
  RA_ERR_ALIGNMENT = -3,     /* pointer or stride violates a 16-byte alignment rule    */
  RA_ERR_WORKSPACE = -4,     /* workspace / packed-weight buffer too small             */
  RA_ERR_CUDA = -5,          /* a CUDA runtime call failed                             */
  RA_ERR_TIMEOUT = -6,       /* a device pipeline wait gave up (see qkv_cte_mx_status) */
  RA_ERR_INDEX = -7          /* reserved: index out of range reported by the host      */
} ra_status;

typedef enum {
  RA_BF16 = 0, RA_FP16 = 1, RA_INT8 = 2, RA_FP32 = 3,
  RA_FP8_E4M3 = 4,   /* OCP FP8 E4M3 (largest finite 448)                          */
  RA_FP8_E5M2 = 5    /* OCP FP8 E5M2 (largest finite 57344)                        */
} ra_dtype;

/* Message of the last failed call on this host thread ("" if none). */
const char* ra_last_error(void);

/* ABI version of this library (bumped on any signature change). */
int32_t ra_abi_version(void);

/* ========================================================================
 * (a) qkv_cte_mx
 * ======================================================================== */

/* Norm selector, after NormType in the page's "Interface" (qk_norm_pre_rope).
 * RMS_ACROSS_HEADS: one RMS per token over the whole segment (Design 1), gamma
 *   [n * head_dim]; applied by the second pass.
 * RMS_PER_HEAD: the upstream qk-norm (Design 1: each head's slice by its own RMS),
 *   gamma [head_dim] shared by the heads; a head fits in one projection tile, so
 *   this norm is applied in the projection epilogue.  Without fused_rope the
 *   segment is then final; with it, the second pass applies the segment's RoPE
 *   (and no norm).  Built for head_dim 64 and 128. */
enum { RA_NORM_NONE = 0, RA_NORM_RMS_ACROSS_HEADS = 1, RA_NORM_RMS_PER_HEAD = 2 };
/* Output layout, after QKVOutputLayout ("Interface", output_layout). */
enum { RA_LAYOUT_BSD = 0, RA_LAYOUT_NBSD = 1 };

typedef struct {
  int64_t B, S;           /* tokens T = B*S; rows of A and of the output             */
  int64_t H;              /* contraction (hidden) size; multiple of 128              */
  int32_t num_heads;      /* Q heads in this call                                     */
  int32_t num_kv_heads;   /* K/V heads; 0 = single-segment call (Design 5)            */
  int32_t head_dim;       /* d_head; multiple of 16                                  */
  int32_t q_norm;         /* RA_NORM_* for the Q segment                              */
  int32_t k_norm;         /* RA_NORM_* for the K segment; must be NONE when num_kv_heads == 0 */
  int32_t fused_rope;     /* 1 = rotate-half RoPE on Q and K; needs cos/sin caches    */
  float norm_eps;         /* epsilon inside the square root                           */
  int32_t output_layout;  /* RA_LAYOUT_BSD: out [B, S, I]; RA_LAYOUT_NBSD: out
                           * [I / head_dim, B, S, head_dim], heads in column order (Q
                           * heads, then K, then V), the layout the page gives the
                           * cross-attention calls ("Interface", output_layout) */
} qkv_cte_mx_params;

/* Size in bytes of the packed weight for an [H, I] MX weight. */
ra_status qkv_cte_mx_packed_weight_bytes(int64_t H, int64_t I, size_t* bytes);

/* One-time weight preparation (not part of the per-token path).
 *   w            [H, I] FP8 E4M3 codes, row-major (the math layout of W).
 *   w_block_exp  [H/32, I] UE8M0 exponents: W_hat[h, i] = e4m3(w[h, i]) * 2^(e[h/32, i]-127)
 *                (MX block of 32 along H).
 *   packed       device buffer of qkv_cte_mx_packed_weight_bytes(H, I) bytes,
 *                16-byte aligned; receives an opaque K-major image of W and its
 *                block scales for the projection kernel.
 * Asynchronous on `stream`.  H % 128 == 0, I % 16 == 0, I <= 2^31-1. */
ra_status qkv_cte_mx_pack_weight(const uint8_t* w, const uint8_t* w_block_exp, int64_t H, int64_t I,
                                 void* packed, size_t packed_bytes, void* stream);

/* Workspace bytes needed by qkv_cte_mx / qkv_cte_mx_project / qkv_cte_mx_norm_rope.
 * The workspace holds a device status word, the per-token sum-of-squares
 * partials (8 bytes per token and 128-column block of Q|K) and one exponent
 * byte per token and 128-column block (see qkv_cte_mx_project).
 * Zero-fill it once after allocation; the calls keep it consistent. */
ra_status qkv_cte_mx_workspace_bytes(const qkv_cte_mx_params* p, size_t* bytes);

/* The whole prologue: projection (with the per-token sums of squares) followed
 * by the across-heads norm + RoPE pass.
 *   a             [T, H] FP8 E4M3 activation codes; 16-byte aligned rows (H % 16 == 0).
 *   a_scale       [T] fp32 per-row dequant scale (the 4-byte tail of the
 *                 page's row-packed [B, S, H+4] activation, passed separately).
 *   w_packed      output of qkv_cte_mx_pack_weight for this H and I.
 *   weight_scales [I] fp32 per-output-channel scale, or NULL (= 1).
 *   bias          [I] bf16, or NULL.
 *   cos_cache, sin_cache  [B, S, head_dim] fp32 rotate-half tables (lanes j and
 *                 j + head_dim/2 pair up); required iff fused_rope.
 *   q_gamma       [num_heads*head_dim] fp32 segment-wide gamma (RMS_ACROSS_HEADS) or
 *                 [head_dim] (RMS_PER_HEAD); required iff q_norm.
 *   k_gamma       likewise for the K segment; required iff k_norm.
 *   out           [T, I] bf16 (BSD), 16-byte aligned.  Q|K|V along the last dim.
 *   workspace     caller-owned, >= qkv_cte_mx_workspace_bytes, 16-byte aligned.
 * Errors: validation codes above; RA_ERR_CUDA on launch failure.  A device
 * wait timeout is reported by qkv_cte_mx_status. */
ra_status qkv_cte_mx(const qkv_cte_mx_params* p, const uint8_t* a, const float* a_scale,
                     const void* w_packed, const float* weight_scales, const uint16_t* bias,
                     const float* cos_cache, const float* sin_cache, const float* q_gamma,
                     const float* k_gamma, uint16_t* out, void* workspace, size_t workspace_bytes,
                     void* stream);

/* First half of qkv_cte_mx on its own: everything that needs no across-heads
 * statistic.  O = dequant(A) @ dequant(W) + bias, the per-token Q / K sums of
 * squares of O (Design 1a) into the workspace, and the segment-wide gamma of
 * each normed segment (Design 1c; inv_rms is one scalar per token and segment
 * and RoPE is linear, so rot(O * inv_rms * gamma) = inv_rms * rot(O * gamma)).
 * Columns the second pass does not touch (V, or everything when norms and RoPE
 * are off -- e.g. the V-only call) are final bf16 in `out`.  Columns it rewrites
 * (Q and/or K when normed or rotated) are held in `out` in an internal encoding
 * until qkv_cte_mx_norm_rope runs: fp16 of O * gamma * 2^-e with a power-of-two
 * e per (token, 128-column block) kept in the workspace, so the intermediate
 * carries 11 significant bits and the only bf16 rounding of Q and K is the
 * final one.  Segments with the per-head norm are normed here, each head by
 * its own RMS and the [head_dim] gamma: without fused_rope they are finished
 * (bf16); with it they are held in the same encoding and qkv_cte_mx_norm_rope
 * rotates them.  Arguments as for qkv_cte_mx (no cos/sin: every rotation is
 * applied by the second pass). */
ra_status qkv_cte_mx_project(const qkv_cte_mx_params* p, const uint8_t* a, const float* a_scale,
                             const void* w_packed, const float* weight_scales, const uint16_t* bias,
                             const float* q_gamma, const float* k_gamma, uint16_t* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Second half on its own (Design 1b, Design 2): reduces the sums of squares
 * left in `workspace` by qkv_cte_mx_project for the same `out` into inv_rms per
 * token and across-heads segment, applies it (per-head segments are already
 * normed) and the rotate-half RoPE (cos/sin required iff fused_rope) to the
 * encoded Q and K columns and writes them back into `out` as bf16.  V is not
 * touched.  This is the seam where a tensor-parallel
 * all-reduce of the sums would go. */
ra_status qkv_cte_mx_norm_rope(const qkv_cte_mx_params* p, const float* cos_cache,
                               const float* sin_cache, uint16_t* out, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Synchronises `stream`, reads the workspace status word, clears it, and
 * stores it in *device_status (0 = fine).  Returns RA_ERR_TIMEOUT if a wait of
 * the projection or of the pipelined norm/RoPE pass gave up since the last
 * read, else RA_OK.  workspace NULL reads the status word of the static
 * workspace that qkv_cte_mx_noalloc uses on the current device. */
ra_status qkv_cte_mx_status(void* workspace, void* stream, int32_t* device_status);

/* qkv_cte_mx for callers that cannot allocate device memory.  The pages have
 * no counterpart; this entry point exists for host code that must not call
 * cudaMalloc where it runs the operator (a plugin of an inference runtime
 * that owns all device memory, or a serving loop that cannot afford
 * cudaMalloc's implicit device synchronisation).  It takes the same arguments
 * as qkv_cte_mx minus the workspace and allocates nothing: its scratch is a
 * static 32 MiB device array inside this library, held on every GPU that
 * loads the library until the process exits.
 *   - Problems whose qkv_cte_mx_workspace_bytes exceeds 32 MiB are rejected
 *     with RA_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and later calls on that
 *     device reuse it.
 *   - Every call shares the array: calls that overlap on the GPU (unordered
 *     streams or threads) race and give undefined results.  Calls ordered on
 *     one stream are independent (each call clears the status word, once its
 *     arguments have passed every check).
 *   - A device wait timeout is recorded in the array's status word; read it
 *     with qkv_cte_mx_status(NULL, stream, &word) after the call and before
 *     the next one, which clears it. */
ra_status qkv_cte_mx_noalloc(const qkv_cte_mx_params* p, const uint8_t* a, const float* a_scale,
                             const void* w_packed, const float* weight_scales, const uint16_t* bias,
                             const float* cos_cache, const float* sin_cache, const float* q_gamma,
                             const float* k_gamma, uint16_t* out, void* stream);

/* Test hook: time limit, in nanoseconds, of each device pipeline wait in the
 * projection kernel, the pipelined norm/RoPE pass and the pipelined KV cache
 * kernel (default 2e9).  Values < 1000 are raised to 1000. */
void ra_set_wait_timeout_ns(int64_t ns);

/* Test hook for host-side checks without a device.  While `on` is non-zero,
 * every entry point returns RA_OK as soon as its arguments have passed the
 * host checks, before any CUDA runtime call: nothing is launched, copied or
 * looked up, and the status readers report 0.  A rejected call is rejected as
 * usual.  Tests that hand the library placeholder addresses set it, so that no
 * such address can reach a kernel whatever the order of the checks.  Global to
 * the process. */
void ra_test_validate_only(int32_t on);

/* Test hook for failure detection.  The next projection launch (qkv_cte_mx or
 * qkv_cte_mx_project) issues none of its TMA loads, so the waits of its
 * pipeline run out after the time limit above; every CTA then records the
 * timeout in the workspace status word, releases its tensor memory and exits,
 * and qkv_cte_mx_status reports RA_ERR_TIMEOUT.  Nothing is in flight when the
 * waits give up, so the CUDA context stays usable.  The output of that launch
 * is undefined.  Applies to one launch, then clears itself. */
void ra_test_stall_next_projection(void);

/* Test hook for failure detection.  The next norm/RoPE pass (qkv_cte_mx or
 * qkv_cte_mx_norm_rope) that runs a pipelined kernel -- head_dim 64 or 128, and
 * BSD output with at most 24 KB of rewritten Q/K columns per token, or NBSd
 * output -- issues none of its copies, so its waits run out after the time
 * limit above; every block
 * records the timeout in the workspace status word and exits, and
 * qkv_cte_mx_status reports RA_ERR_TIMEOUT.  Nothing is in flight when the
 * waits give up.  The output of that call is undefined.  Applies to one call,
 * then clears itself. */
void ra_test_stall_next_norm_rope(void);

/* ========================================================================
 * Row FP8 quantisation of the activation (the step before qkv_cte_mx)
 * ======================================================================== */

/* AWS Neuron "Kernel reference: qkv_cte", section "Interface": the projection's
 * input is a row-packed activation -- H FP8 (E4M3) codes followed by a 4-byte
 * fp32 dequantisation scale per row -- made by a row quantiser from the bf16
 * hidden state.  The page gives no formula; this library computes, per row t,
 * with the code defined by the layout's dequantisation identity x ~ code * scale,
 *   m = max(max_h |x[t,h]|, 2^-100),  scale[t] = m / 448,
 *   code[t,h] = E4M3(x[t,h] / scale[t]),
 * every step in fp32 rounded to nearest-even (the divisions correctly rounded),
 * the E4M3 rounding half-to-even and saturated to +-448 (the sign of zero is
 * kept); the floor keeps the scale a normal fp32 number for rows of zeros or of
 * bf16 subnormals.  Inputs must be finite.
 *
 * row_quantize_e4m3: the split form qkv_cte_mx reads (`a` and `a_scale`).
 *   x      [T, H] bf16 bit patterns, device, 16-byte aligned
 *   codes  [T, H] E4M3 codes, device, 8-byte aligned (written)
 *   scale  [T] fp32 dequantisation scales, device, 4-byte aligned (written)
 * row_quantize_e4m3_packed: the page's row-packed layout.
 *   packed [T, H + 4] bytes, device, 4-byte aligned (written): row t holds its H
 *          codes, then its scale as a little-endian IEEE binary32.
 * T >= 1; H a positive multiple of 8.  All buffers are caller-owned; the call is
 * asynchronous on `stream` and allocates nothing.  Errors: RA_ERR_INVALID_ARG
 * (NULL pointer, bad size), RA_ERR_ALIGNMENT, RA_ERR_CUDA (launch failure). */
ra_status row_quantize_e4m3(const uint16_t* x, int64_t T, int64_t H, uint8_t* codes, float* scale,
                            void* stream);
ra_status row_quantize_e4m3_packed(const uint16_t* x, int64_t T, int64_t H, uint8_t* packed,
                                   void* stream);

/* ========================================================================
 * (b) kv_rms_norm_rope_cache
 * ======================================================================== */

/* cache_mode, from the page's cache/index constraint table:
 *   NORM        caches [B, N, cache_seq_len, D]; index [B, S] holds each token's
 *               offset in its batch's cache (values may repeat across batches).
 *   PA          caches [block_num, block_size, N, D]; index [B*S], one slot per token.
 *   PA_BNSD     caches [block_num, N, block_size, D]; index [B*S], one slot per token.
 *   PA_BLK_BNSD caches as PA_BNSD; index [B * ceil(S / block_size)] holds the start
 *               slot of each block of block_size tokens: token s of batch b goes to
 *               index[b, s / block_size] + s % block_size (-1 skips the block).
 *   PA_NZ, PA_BLK_NZ (FRACTAL_NZ layouts for Ascend's cube unit): RA_ERR_UNSUPPORTED. */
enum { RA_CACHE_NORM = 0, RA_CACHE_PA = 1, RA_CACHE_PA_BNSD = 2, RA_CACHE_PA_NZ = 3,
       RA_CACHE_PA_BLK_BNSD = 4, RA_CACHE_PA_BLK_NZ = 5 };

typedef struct {
  int64_t B, N, S;        /* kv is [B, N, S, Dkv]                                     */
  int64_t Dkv;            /* last dim of kv                                           */
  int64_t Dv;             /* V1: rms_size (= Dkv - rope_size); V2: last dim of v_optional */
  int32_t rope_size;      /* RoPE width (64 in both of the page's modes); even        */
  int32_t variant;        /* 1 = V1 combined kv (N == 1), 2 = V2 separate kv (N in 1,2,4,8) */
  int32_t cache_mode;     /* RA_CACHE_*                                               */
  int64_t block_num;      /* paged cache blocks (PA modes)                            */
  int64_t block_size;     /* slots per block (PA modes); %16 for 2-byte caches, %32 for
                           * 1-byte caches (both when the two caches differ)          */
  int32_t kv_dtype;       /* RA_BF16 or RA_FP16 (kv, gamma, cos, sin, v_optional share it) */
  int32_t k_cache_dtype;  /* = kv_dtype, or RA_INT8 / RA_FP8_E4M3 / RA_FP8_E5M2 when
                           * k_rope_scale is given                                    */
  int32_t ckv_cache_dtype;/* likewise with c_kv_scale                                  */
  float epsilon;          /* RMSNorm epsilon (page default 1e-5)                      */
  int32_t is_output_kv;   /* 1 = also write k_rope and c_kv (in NORM mode only for V2
                           * with quantisation, per the page's combination table)    */
  int32_t rope_s_broadcast;  /* 1 = cos/sin are [B, N, 1, rope_size], broadcast over S */
  int64_t cache_seq_len;  /* NORM mode: Scache (>= S); ignored otherwise             */
  int32_t k_quant_scalar; /* V1: 1 = k_rope_scale / k_rope_offset are [1] (one value for
                           * every channel) instead of [k_w]; must be 0 in V2         */
  int32_t c_kv_quant_scalar; /* V1: likewise for c_kv_scale / c_kv_offset             */
} kv_rms_norm_rope_cache_params;

/* One call of KvRmsNormRopeCache.
 *   kv          [B, N, S, Dkv] bf16 or fp16 (kv_dtype).
 *   gamma       [rms_size] (rms_size = Dkv - rope_size in V1, Dkv in V2).
 *   cos, sin    [B, N, S, rope_size], or [B, N, 1, rope_size] with rope_s_broadcast
 *               (interleaved-RoPE tables).
 *   index       int64, shaped by cache_mode (see RA_CACHE_*); -1 = skip.  Slots
 *               (PA modes: block starts / block_size) must be unique.
 *   k_cache     paged cache of width k_w = rope_size (V1) or Dkv (V2), updated in place.
 *   ckv_cache   paged cache of width c_w = rms_size (V1) or Dv (V2), updated in place.
 *   k_rope_scale / k_rope_offset  fp32 per channel: [k_w] (V1; [1] with k_quant_scalar)
 *               or [N, k_w] (V2); NULL = absent.
 *   c_kv_scale   / c_kv_offset    fp32 per channel: [c_w] (V1; [1] with c_kv_quant_scalar)
 *               or [N, c_w] (V2); NULL = absent.
 *               An offset without its scale is rejected.
 *   v_optional  [B, N, S, Dv] bf16; required in V2, must be NULL in V1.
 *   k_rope      [B, N, S, k_w] and c_kv [B, N, S, c_w], kv_dtype: written iff outputs
 *               are on (see is_output_kv).
 *   Quantised caches hold round_half_even(x * scale + offset) clamped to [-128, 127]
 *   (int8, formula (3)), or x * scale + offset rounded to the nearest FP8 value,
 *   ties to even, saturated at the largest finite value (FP8 caches).
 *   dev_error_count  optional int32 device counter: incremented once per token whose
 *               slot lies outside the cache (any negative index other than -1, or
 *               beyond block_num*block_size / cache_seq_len); such tokens are not written.
 * V1 in NORM mode takes no quantisation parameters.
 * All row pointers 16-byte aligned; Dkv, Dv and rope_size multiples of 8.
 * Calls of the two common row shapes (V1 Dkv 576 with rope_size 64; V2 Dkv 192,
 * Dv 128, rope_size 64) in PA / PA_BNSD mode with int8 or 16-bit caches and
 * per-token cos/sin run a pipelined kernel whose waits have a time limit; a
 * wait that runs out is reported by kv_rms_norm_rope_cache_status.  The first
 * call on each device looks up that status word (cudaGetSymbolAddress); make
 * it before any stream capture. */
ra_status kv_rms_norm_rope_cache(const kv_rms_norm_rope_cache_params* p, const uint16_t* kv,
                                 const uint16_t* gamma, const uint16_t* cos, const uint16_t* sin,
                                 const int64_t* index, void* k_cache, void* ckv_cache,
                                 const float* k_rope_scale, const float* c_kv_scale,
                                 const float* k_rope_offset, const float* c_kv_offset,
                                 const uint16_t* v_optional, uint16_t* k_rope, uint16_t* c_kv,
                                 int32_t* dev_error_count, void* stream);

/* Synchronises `stream`, reads this library's KV status word on the current
 * device, clears it, and stores it in *device_status (0 = fine).  Returns
 * RA_ERR_TIMEOUT if a pipeline wait of kv_rms_norm_rope_cache gave up since the
 * last read (that call's caches and outputs are then undefined), else RA_OK.
 * The word is shared by every call on the device. */
ra_status kv_rms_norm_rope_cache_status(void* stream, int32_t* device_status);

/* Test hook for failure detection.  The next kv_rms_norm_rope_cache call that
 * runs the pipelined kernel (see above) issues none of its copies, so its waits
 * run out after the time limit of ra_set_wait_timeout_ns; every block records
 * the timeout in the status word and exits, and kv_rms_norm_rope_cache_status
 * reports RA_ERR_TIMEOUT.  Nothing is in flight when the waits give up.  The
 * caches of that call are undefined.  Applies to one call, then clears itself. */
void ra_test_stall_next_kv_cache(void);

#ifdef __cplusplus
}
#endif
#endif /* ROPE_ATTENTION_H_ */
