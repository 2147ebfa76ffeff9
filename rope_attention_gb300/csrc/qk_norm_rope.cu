// K2: across-heads RMSNorm + rotate-half RoPE, applied in place to Q and K.
//
// AWS Neuron "Kernel reference: qkv_cte", Design 1b-1c and Design 2:
//   inv_rms[t] = rsqrt(sum_sq[t] / (n_heads * d_head) + eps), one per token and
//                segment (tp = 1, so the sums are complete on this GPU);
//   y          = x * inv_rms * gamma          (segment-wide gamma, per channel);
//   out_lo     = y_lo * cos_lo - y_hi * sin_lo,  out_hi = y_hi * cos_hi + y_lo * sin_hi,
//                lanes (j, j + d/2) of every head, cos/sin shared by all heads.
// The un-normalised Q|K columns arrive in ``out`` as fp16 of v * 2^-e, with one
// power-of-two exponent per (token, 128-column block) in the workspace: 11
// significant bits in 2 bytes, so the only bf16 rounding is the final one;
// V is never touched.  The per-token sums arrive as per-column-tile partials
// written by the projection epilogue; they are reduced here in a fixed order,
// so the result is deterministic.
//
// GB300 mapping: HBM-bound stream over Q|K.  A block owns kTok tokens; each
// thread owns fixed (head, lane-group) items, keeps their gamma in registers
// and walks the block's tokens, moving 16-byte vectors (8 bf16) of the low and
// high half of its head together so the rotation needs no shuffle.
#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int kThreads = 256;
constexpr int kTok = 8;

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = bf16_lo(w[k]);
    f[2 * k + 1] = bf16_hi(w[k]);
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  u.z = pack_bf16x2(f[4], f[5]);
  u.w = pack_bf16x2(f[6], f[7]);
  return u;
}
__device__ __forceinline__ void load8f(const float* p, float (&f)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// 8 values of the projection's scaled fp16 encoding: fp16 code * 2^e
__device__ __forceinline__ void load8h(const uint16_t* p, float up, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
    f[2 * k] = t.x * up;
    f[2 * k + 1] = t.y * up;
  }
}
__device__ __forceinline__ float block_up(const NormRopeLaunch& p, int64_t t, int64_t col) {
  return exp2_int(p.exps[static_cast<size_t>(col / kPartCols) * p.T + t]);
}

__global__ void __launch_bounds__(kThreads) qk_norm_rope_kernel(const NormRopeLaunch p) {
  __shared__ float s_inv[kTok][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTok;
  const int ntok = static_cast<int>(p.T - t0 < kTok ? p.T - t0 : kTok);
  const int d = p.head_dim, half = d / 2;
  const int nq = p.num_q_heads, nk = p.num_k_heads;

  if (warp < kTok) {
    const int64_t t = t0 + warp;
    float sq = 0.f, sk = 0.f;
    if (warp < ntok) {
      for (int j = lane; j < p.n_part_tiles; j += 32) {
        const float2 v = p.partials[static_cast<size_t>(j) * p.T + t];
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
      s_inv[warp][0] = p.q_norm ? rsqrtf(sq / static_cast<float>(nq * d) + p.eps) : 1.f;
      s_inv[warp][1] = p.k_norm ? rsqrtf(sk / static_cast<float>(nk * d) + p.eps) : 1.f;
    }
  }
  __syncthreads();

  const bool do_q = p.q_norm || p.rope;
  const bool do_k = nk > 0 && (p.k_norm || p.rope);
  const int h_begin = do_q ? 0 : nq;
  const int h_end = do_k ? nq + nk : nq;
  const int per_head = p.rope ? half / 8 : d / 8;
  const int items = (h_end - h_begin) * per_head;

  for (int it = threadIdx.x; it < items; it += kThreads) {
    const int hh = h_begin + it / per_head;
    const int u = it % per_head;
    const bool is_k = hh >= nq;
    const int hseg = is_k ? hh - nq : hh;
    const float* gamma = is_k ? (p.k_norm ? p.k_gamma : nullptr) : (p.q_norm ? p.q_gamma : nullptr);
    const int64_t col = static_cast<int64_t>(hh) * d + 8 * u;
    if (p.rope) {
      float glo[8], ghi[8];
      if (gamma != nullptr) {
        load8f(gamma + hseg * d + 8 * u, glo);
        load8f(gamma + hseg * d + half + 8 * u, ghi);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) glo[j] = ghi[j] = 1.f;
      }
#pragma unroll 2
      for (int tl = 0; tl < ntok; ++tl) {
        const int64_t t = t0 + tl;
        uint16_t* row = p.out + t * p.I;
        float xlo[8], xhi[8], clo[8], chi[8], slo[8], shi[8];
        load8h(row + col, block_up(p, t, col), xlo);
        load8h(row + col + half, block_up(p, t, col + half), xhi);
        const float* cs = p.cos + t * d + 8 * u;
        const float* sn = p.sin + t * d + 8 * u;
        load8f(cs, clo);
        load8f(cs + half, chi);
        load8f(sn, slo);
        load8f(sn + half, shi);
        const float inv = s_inv[tl][is_k ? 1 : 0];
        float olo[8], ohi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float ylo = xlo[j] * inv * glo[j];
          const float yhi = xhi[j] * inv * ghi[j];
          olo[j] = ylo * clo[j] - yhi * slo[j];
          ohi[j] = yhi * chi[j] + ylo * shi[j];
        }
        *reinterpret_cast<uint4*>(row + col) = pack8(olo);
        *reinterpret_cast<uint4*>(row + col + half) = pack8(ohi);
      }
    } else {
      float g[8];
      if (gamma != nullptr) {
        load8f(gamma + hseg * d + 8 * u, g);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = 1.f;
      }
#pragma unroll 2
      for (int tl = 0; tl < ntok; ++tl) {
        const int64_t t = t0 + tl;
        uint16_t* row = p.out + t * p.I;
        float x[8];
        load8h(row + col, block_up(p, t, col), x);
        const float inv = s_inv[tl][is_k ? 1 : 0];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = x[j] * inv * g[j];
        *reinterpret_cast<uint4*>(row + col) = pack8(x);
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
