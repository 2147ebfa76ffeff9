// Row FP8 quantisation of the activation: bf16 [T, H] -> E4M3 codes + one fp32
// dequantisation scale per row, split ([T, H] codes and [T] scales, the form the
// projection reads) or in the row-packed [T, H + 4] layout.
//
// AWS Neuron "Kernel reference: qkv_cte", section "Interface": the projection's
// input is the row-packed activation, H FP8 codes followed by a 4-byte fp32
// dequantisation scale per row, made by a row quantiser from the bf16 hidden
// state.  The page gives no formula; the plain absmax reading is used, with the
// code defined by the layout's dequantisation identity x ~ code * scale:
//   m = max(max_h |x|, 2^-100),  scale = m / 448,  code = E4M3(x / scale),
// every step in fp32 with round-to-nearest-even (the division correctly
// rounded), the E4M3 rounding half-to-even with saturation to +-448 (the floor
// keeps the scale a normal fp32 number for rows of zeros or of bf16 subnormals).
//
// GB300 mapping: an HBM stream (2 bytes in, 1 byte out per element).  One warp
// per row, persistent over rows: the row is loaded once into registers with
// 16-byte loads, its amax is taken on the bf16 bit patterns (|x| as an unsigned
// 15-bit integer orders like the value) with per-halfword max and one
// warp-wide integer max-reduction, then each lane turns its chunks into
// quotients |x| / scale (below), converts them with the hardware E4M3x2
// conversion, puts the signs of x back on the codes, and writes 8 bytes per
// chunk, coalesced across the warp.  Rows longer than the register budget
// (H > 8192) take a two-pass path that re-reads the row (from L2).
//
// The division.  A per-element IEEE division costs more instructions than the
// HBM stream leaves room for, so the row's divisor is inverted once,
// r = RN(1 / scale), and each quotient is q0 = RN(|x| * r) followed by one
// remainder correction, q = RN(q0 + RN(|x| - q0 * scale) * r) with fused
// multiply-adds (the correction step of P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990).  q itself can differ from the correctly rounded quotient in its last
// bit where the remainder underflows, but the codes cannot: every input the
// quantiser can meet was enumerated -- each row maximum m (every positive finite
// bf16 value >= 2^-100, the floor included) with every bf16 magnitude |x| <= m,
// 526.7 million pairs -- and E4M3(q) equals E4M3(RN(|x| / scale)) on all of
// them, while E4M3(RN(|x| * r)) alone differs on 31920.
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"
#include "row_quant.h"

namespace ra {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kE4m3Max = 448.f;
constexpr float kAmaxFloor = 7.88860905e-31f;  // 2^-100, exact in fp32

__device__ __forceinline__ uint32_t abs_max_bits(uint32_t m, uint4 v) {
  m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
  return __vmaxu2(m, v.w & 0x7FFF7FFFu);
}

// the row's amax as a float, reduced over the warp
__device__ __forceinline__ float warp_amax(uint32_t m) {
  uint32_t mm = max(m & 0xFFFFu, m >> 16);
  mm = __reduce_max_sync(0xffffffffu, mm);
  return __uint_as_float(mm << 16);
}

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// The row's divisor: scale, -scale and RN(1 / scale), each as a pair for the
// packed fp32x2 arithmetic
struct RowDiv {
  float2 s, neg_s, r;
};

__device__ __forceinline__ RowDiv row_divisor(float amax, float& scale) {
  scale = __fdiv_rn(fmaxf(amax, kAmaxFloor), kE4m3Max);
  const float r = __frcp_rn(scale);
  return {make_float2(scale, scale), make_float2(-scale, -scale), make_float2(r, r)};
}

// |x| / scale for a bf16 pair: q0 = |x| * r, then one remainder correction
__device__ __forceinline__ float2 quot2(uint32_t bf16x2, const RowDiv& d) {
  const float2 a = bf16x2_to_float2(bf16x2 & 0x7FFF7FFFu);
  const float2 q0 = __fmul2_rn(a, d.r);
  const float2 rem = __ffma2_rn(q0, d.neg_s, a);  // exact |x| - q0 * scale (or underflowed)
  return __ffma2_rn(rem, d.r, q0);
}

// the sign bits of four bf16 values (two words), at the top of each code byte
__device__ __forceinline__ uint32_t signs4(uint32_t lo, uint32_t hi) {
  return __byte_perm(lo, hi, 0x7531) & 0x80808080u;
}

// 8 codes (two 32-bit words, first element in the lowest byte) for one chunk
__device__ __forceinline__ uint2 quant8(uint4 v, const RowDiv& d) {
  const float2 f0 = quot2(v.x, d), f1 = quot2(v.y, d);
  const float2 f2 = quot2(v.z, d), f3 = quot2(v.w, d);
  return make_uint2((e4m3x2(f0.x, f0.y) | (e4m3x2(f1.x, f1.y) << 16)) | signs4(v.x, v.y),
                    (e4m3x2(f2.x, f2.y) | (e4m3x2(f3.x, f3.y) << 16)) | signs4(v.z, v.w));
}

__device__ __forceinline__ void store8(uint8_t* dst, uint2 c, bool packed) {
  if (packed) {  // packed rows are only 4-byte aligned (H + 4 bytes apart)
    reinterpret_cast<uint32_t*>(dst)[0] = c.x;
    reinterpret_cast<uint32_t*>(dst)[1] = c.y;
  } else {
    *reinterpret_cast<uint2*>(dst) = c;
  }
}

// CPL = 16-byte chunks per lane held in registers; CPL == 0: two-pass path for any H
template <int CPL, bool PACKED>
__global__ void __launch_bounds__(kThreads) row_quant_kernel(const uint16_t* __restrict__ x, int64_t T,
                                                             int H, uint8_t* __restrict__ codes,
                                                             float* __restrict__ scale,
                                                             int64_t out_stride) {
  const int lane = threadIdx.x & 31;
  const int chunks = H / 8;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); row < T;
       row += warps) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * H);
    uint8_t* cr = codes + row * out_stride;
    float sc;
    if constexpr (CPL > 0) {
      uint4 v[CPL];
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        v[i] = c < chunks ? __ldcs(xr + c) : make_uint4(0, 0, 0, 0);
        m = abs_max_bits(m, v[i]);
      }
      const RowDiv d = row_divisor(warp_amax(m), sc);
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < chunks) store8(cr + 8 * c, quant8(v[i], d), PACKED);
      }
    } else {
      uint32_t m = 0;
      for (int c = lane; c < chunks; c += 32) m = abs_max_bits(m, __ldg(xr + c));
      const RowDiv d = row_divisor(warp_amax(m), sc);
      for (int c = lane; c < chunks; c += 32) store8(cr + 8 * c, quant8(__ldcs(xr + c), d), PACKED);
    }
    if (lane == 0) {
      if (PACKED) *reinterpret_cast<float*>(cr + H) = sc;
      else scale[row] = sc;
    }
  }
}

template <int CPL, bool PACKED>
cudaError_t launch_one(const uint16_t* x, int64_t T, int H, uint8_t* codes, float* scale,
                       int64_t out_stride, cudaStream_t st) {
  auto kernel = row_quant_kernel<CPL, PACKED>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (T + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(per_sm) * device_sm_count();
  kernel<<<static_cast<unsigned>(want < cap ? want : cap), kThreads, 0, st>>>(x, T, H, codes, scale,
                                                                            out_stride);
  return cudaGetLastError();
}

template <bool PACKED>
cudaError_t launch_rows(const uint16_t* x, int64_t T, int H, uint8_t* codes, float* scale,
                        int64_t out_stride, cudaStream_t st) {
  const int need = (H / 8 + 31) / 32;  // chunks per lane
  if (need <= 1) return launch_one<1, PACKED>(x, T, H, codes, scale, out_stride, st);
  if (need <= 2) return launch_one<2, PACKED>(x, T, H, codes, scale, out_stride, st);
  if (need <= 4) return launch_one<4, PACKED>(x, T, H, codes, scale, out_stride, st);
  if (need <= 8) return launch_one<8, PACKED>(x, T, H, codes, scale, out_stride, st);
  if (need <= 12) return launch_one<12, PACKED>(x, T, H, codes, scale, out_stride, st);
  if (need <= 16) return launch_one<16, PACKED>(x, T, H, codes, scale, out_stride, st);
  if (need <= 20) return launch_one<20, PACKED>(x, T, H, codes, scale, out_stride, st);
  if (need <= 24) return launch_one<24, PACKED>(x, T, H, codes, scale, out_stride, st);
  if (need <= 32) return launch_one<32, PACKED>(x, T, H, codes, scale, out_stride, st);
  return launch_one<0, PACKED>(x, T, H, codes, scale, out_stride, st);
}

}  // namespace

cudaError_t launch_row_quantize(const uint16_t* x, int64_t T, int64_t H, uint8_t* codes, float* scale,
                                bool packed, cudaStream_t stream) {
  const int h = static_cast<int>(H);
  return packed ? launch_rows<true>(x, T, h, codes, nullptr, H + 4, stream)
                : launch_rows<false>(x, T, h, codes, scale, H, stream);
}

}  // namespace ra
