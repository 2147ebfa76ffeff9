// K2: the across-heads part of the RMSNorm and the rotate-half RoPE, written
// in place into Q and K.
//
// AWS Neuron "Kernel reference: qkv_cte", Design 1b-1c and Design 2:
//   inv_rms[t] = rsqrt(sum_sq[t] / (n_heads * d_head) + eps), one per token and
//                segment (tp = 1, so the sums are complete on this GPU);
//   y          = x * inv_rms * gamma          (segment-wide gamma, per channel);
//   out_lo     = y_lo * cos_lo - y_hi * sin_lo,  out_hi = y_hi * cos_hi + y_lo * sin_hi,
//                lanes (j, j + d/2) of every head, cos/sin shared by all heads.
// The projection has already multiplied by gamma (a per-channel factor, which
// commutes with the per-token inv_rms and with the rotation) and stored Q/K as
// fp16 codes with a power-of-two exponent per (token, 128-column block), so this
// pass computes out = rot(code * 2^e * inv_rms) and rounds once, to bf16.  The
// per-token sums arrive as per-128-column-block partials written by the
// projection epilogue; they are reduced here in a fixed order, so the result
// is deterministic.  V is never touched.
//
// GB300 mapping: an HBM-bound stream (2 bytes read + 2 written per element)
// with no block-wide synchronisation in its main loop.  A block owns 8 tokens:
// its warps first reduce the tokens' partial sums (contiguous per token), then
// each thread owns fixed 8-column items (the low and high half of a head move
// together, so the rotation needs no shuffle) and walks the tokens two at a
// time so that several 16-byte loads are in flight; cos/sin loads are warp
// broadcasts (all heads of a token share them); the arithmetic uses packed
// fp32x2 FMAs; the bf16 results are 16-byte vectors, coalesced across threads.
#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int kThreads = 128;
constexpr int kTok = 8;        // tokens per block
constexpr int kUnroll = 2;     // tokens whose loads are in flight together per item

__device__ __forceinline__ void ldg8f(const float* p, float2 (&f)[4]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = make_float2(a.x, a.y); f[1] = make_float2(a.z, a.w);
  f[2] = make_float2(b.x, b.y); f[3] = make_float2(b.z, b.w);
}
// 8 values of the projection's encoding (fp16 code * 2^e), times `s`
__device__ __forceinline__ void decode8(uint4 u, float s, float2 (&f)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  const float2 ss = make_float2(s, s);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    f[k] = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&w[k])), ss);
}
__device__ __forceinline__ uint4 pack8(const float2 (&f)[4]) {
  uint4 u;
  u.x = pack_bf16x2(f[0].x, f[0].y);
  u.y = pack_bf16x2(f[1].x, f[1].y);
  u.z = pack_bf16x2(f[2].x, f[2].y);
  u.w = pack_bf16x2(f[3].x, f[3].y);
  return u;
}

__global__ void __launch_bounds__(kThreads) qk_norm_rope_kernel(const NormRopeLaunch p) {
  __shared__ float s_inv[kTok][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTok;
  const int ntok = static_cast<int>(p.T - t0 < kTok ? p.T - t0 : kTok);
  const int d = p.head_dim, half = d / 2;
  const int nq = p.num_q_heads, nk = p.num_k_heads;
  const bool do_q = p.do_q != 0;
  const bool do_k = nk > 0 && p.do_k != 0;
  const int h_begin = do_q ? 0 : nq;
  const int h_end = do_k ? nq + nk : nq;
  const int q_end = nq * d;
  const bool rotate = p.rope != 0;
  // item = 8 columns; a rotating item also carries the 8 columns half a head away
  const int per_head = rotate ? half / 8 : d / 8;
  const int items = (h_end - h_begin) * per_head;

  // 1b: inv_rms per token, from its partial sums in a fixed order
  for (int tl = warp; tl < kTok; tl += kThreads / 32) {
    float sq = 0.f, sk = 0.f;
    if (tl < ntok) {
      const float2* pa = p.partials + (t0 + tl) * p.part_stride;
      for (int j = lane; j < p.n_part_tiles; j += 32) {
        const float2 v = __ldg(pa + j);
        sq += v.x;
        sk += v.y;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (lane == 0) {
      s_inv[tl][0] = p.q_norm ? rsqrtf(sq / static_cast<float>(nq * d) + p.eps) : 1.f;
      s_inv[tl][1] = p.k_norm ? rsqrtf(sk / static_cast<float>(nk * d) + p.eps) : 1.f;
    }
  }
  __syncthreads();

  // each thread owns items (column offsets fixed for the block) and walks the
  // block's tokens, kUnroll at a time so that several 16-byte loads are in flight
  for (int it = threadIdx.x; it < items; it += kThreads) {
    const int u = it % per_head;
    const int col = (h_begin + it / per_head) * d + 8 * u;
    const int seg = col < q_end ? 0 : 1;
    const int blk_lo = col / kPartCols, blk_hi = (col + half) / kPartCols;
    const int jc = rotate ? 8 * u : 0;  // lane of the head for cos/sin
    // where token t's columns [col, col + 8) live: BSD [T, I], or NBSd [I / d, T, d]
    const int64_t base = p.nbsd ? static_cast<int64_t>(col / d) * p.T * d + col % d : col;
    const int64_t tstride = p.nbsd ? d : p.I;
    for (int tb = 0; tb < ntok; tb += kUnroll) {
      uint4 cl[kUnroll], ch[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (tb + k < ntok) {
          const uint16_t* src = p.out + (t0 + tb + k) * tstride + base;
          cl[k] = __ldcs(reinterpret_cast<const uint4*>(src));
          if (rotate) ch[k] = __ldcs(reinterpret_cast<const uint4*>(src + half));
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (tb + k >= ntok) break;
        const int64_t t = t0 + tb + k;
        const int8_t* ex = p.exps + t * p.exp_stride;
        const float inv = s_inv[tb + k][seg];
        uint16_t* dst = p.out + t * tstride + base;
        float2 y_lo[4];
        decode8(cl[k], inv * exp2_int(ex[blk_lo]), y_lo);
        if (rotate) {
          float2 y_hi[4], c_lo[4], c_hi[4], s_lo[4], s_hi[4];
          decode8(ch[k], inv * exp2_int(ex[blk_hi]), y_hi);
          const float* cs = p.cos + t * d + jc;
          const float* sn = p.sin + t * d + jc;
          ldg8f(cs, c_lo);
          ldg8f(cs + half, c_hi);
          ldg8f(sn, s_lo);
          ldg8f(sn + half, s_hi);
          float2 o_lo[4], o_hi[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            o_lo[m] = __ffma2_rn(y_lo[m], c_lo[m], __fmul2_rn(y_hi[m], make_float2(-s_lo[m].x, -s_lo[m].y)));
            o_hi[m] = __ffma2_rn(y_hi[m], c_hi[m], __fmul2_rn(y_lo[m], s_hi[m]));
          }
          *reinterpret_cast<uint4*>(dst) = pack8(o_lo);
          *reinterpret_cast<uint4*>(dst + half) = pack8(o_hi);
        } else {
          *reinterpret_cast<uint4*>(dst) = pack8(y_lo);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_qk_norm_rope(const NormRopeLaunch& L, cudaStream_t stream) {
  const int64_t blocks = (L.T + kTok - 1) / kTok;
  qk_norm_rope_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(L);
  return cudaGetLastError();
}

}  // namespace ra
