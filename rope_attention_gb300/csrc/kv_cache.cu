// K3: KvRmsNormRopeCache -- RMSNorm, interleaved RoPE, optional int8
// quantisation and the index scatter into paged K / CKV caches.
//
// CANN ops-transformer "KvRmsNormRopeCache", formulas (1)-(5):
//  (1) y = x / sqrt(mean(x^2) + eps) * gamma over x = kv[..., :rms_size];
//  (2) x1 = r[0::2], x2 = r[1::2]; y_rope = cat(x1, x2) * cos + cat(-x2, x1) * sin
//      on r = kv[..., Dv:] (V1) or y[..., :rope_size] (V2);
//      rope_out = y_rope (V1) or cat(y_rope, y[..., rope_size:]) (V2);
//  (3) q = round(x * scale + offset).clamp(-128, 127) when a scale is given;
//  (4) k_cache[index[b*S+s]] = Quant(rope_out), ckv_cache[...] = Quant(y) (V1)
//      or Quant(v_optional) (V2); index -1 is skipped;
//  (5) k_rope = rope_out, c_kv = y (V1) / v_optional (V2) when is_output_kv.
// Quantisation uses the fp32 value (before any bf16 rounding); round() is
// round-half-to-even.
//
// GB300 mapping: persistent warps, each walking (b, n, s) rows with a stride of
// the whole grid and loading the next row's data while it processes the current
// one (the op is latency-bound otherwise: a row is only 0.6-1.4 KB).  Every lane moves 16-byte chunks
// (8 bf16); the RMS reduction is a warp shuffle tree; lane l < rope_size/8
// owns interleaved pairs 4l..4l+3, whose outputs land at positions 4l and
// rope_size/2 + 4l of the de-interleaved result, written as 8-byte (bf16) or
// 4-byte (int8) stores.  Cache rows are contiguous, so each scattered slot is
// written with whole 16-byte vectors.
#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = bf16_lo(w[k]);
    f[2 * k + 1] = bf16_hi(w[k]);
  }
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  u.z = pack_bf16x2(f[4], f[5]);
  u.w = pack_bf16x2(f[6], f[7]);
  return u;
}
__device__ __forceinline__ int q8(float v, float scale, float offset) {
  const int q = __float2int_rn(fmaf(v, scale, offset));
  return min(127, max(-128, q));
}
__device__ __forceinline__ uint32_t pack_i8x4(int a, int b, int c, int d) {
  return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8) |
         ((static_cast<uint32_t>(c) & 0xFFu) << 16) | ((static_cast<uint32_t>(d) & 0xFFu) << 24);
}

// n values starting at channel `ch` of a cache row: int8 (quantised) or bf16
template <bool QUANT, int NV>
__device__ __forceinline__ void store_vals(void* row_base, int ch, const float* v, const float* scale,
                                           const float* offset) {
  if constexpr (QUANT) {
    float sc[NV], of[NV];
#pragma unroll
    for (int j = 0; j < NV; j += 4) {
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(scale + ch + j));
      sc[j] = s4.x; sc[j + 1] = s4.y; sc[j + 2] = s4.z; sc[j + 3] = s4.w;
      if (offset != nullptr) {
        const float4 o4 = __ldg(reinterpret_cast<const float4*>(offset + ch + j));
        of[j] = o4.x; of[j + 1] = o4.y; of[j + 2] = o4.z; of[j + 3] = o4.w;
      } else {
        of[j] = of[j + 1] = of[j + 2] = of[j + 3] = 0.f;
      }
    }
    int8_t* dst = static_cast<int8_t*>(row_base) + ch;
    if constexpr (NV == 8) {
      uint2 w;
      w.x = pack_i8x4(q8(v[0], sc[0], of[0]), q8(v[1], sc[1], of[1]), q8(v[2], sc[2], of[2]),
                      q8(v[3], sc[3], of[3]));
      w.y = pack_i8x4(q8(v[4], sc[4], of[4]), q8(v[5], sc[5], of[5]), q8(v[6], sc[6], of[6]),
                      q8(v[7], sc[7], of[7]));
      *reinterpret_cast<uint2*>(dst) = w;
    } else {
      *reinterpret_cast<uint32_t*>(dst) =
          pack_i8x4(q8(v[0], sc[0], of[0]), q8(v[1], sc[1], of[1]), q8(v[2], sc[2], of[2]),
                    q8(v[3], sc[3], of[3]));
    }
  } else {
    uint16_t* dst = static_cast<uint16_t*>(row_base) + ch;
    if constexpr (NV == 8) {
      *reinterpret_cast<uint4*>(dst) = pack8(v);
    } else {
      uint2 w;
      w.x = pack_bf16x2(v[0], v[1]);
      w.y = pack_bf16x2(v[2], v[3]);
      *reinterpret_cast<uint2*>(dst) = w;
    }
  }
}

// Everything one row needs from HBM, loaded as raw 16/8-byte vectors so the
// next row's loads can be in flight while the current row is processed.
template <int CPL>
struct RowIn {
  uint4 x[CPL];            // chunks lane + 32 i of the RMSNorm part of kv
  uint4 xr;                // V1: the lane's chunk of the raw RoPE part
  uint4 v[CPL];            // V2: chunks lane + 32 i of v_optional
  uint2 c1, c2, s1, s2;    // cos/sin for pairs 4l..4l+3 at j and R/2 + j
  int64_t slot;
};

template <int VARIANT, int CPL>
__device__ __forceinline__ void load_row(const KvLaunch& p, int64_t row, int lane, int rms,
                                         int rms_chunks, int v_chunks, int rope_lanes,
                                         RowIn<CPL>& in) {
  const uint16_t* x = p.kv + row * p.Dkv;
  const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = lane + 32 * i;
    in.x[i] = c < rms_chunks ? __ldcs(reinterpret_cast<const uint4*>(x + 8 * c)) : z;
  }
  if (VARIANT == 1)
    in.xr = lane < rope_lanes ? __ldcs(reinterpret_cast<const uint4*>(x + rms + 8 * lane)) : z;
  if (VARIANT == 2) {
    const uint16_t* vrow = p.v + row * p.Dv;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      in.v[i] = c < v_chunks ? __ldcs(reinterpret_cast<const uint4*>(vrow + 8 * c)) : z;
    }
  }
  if (lane < rope_lanes) {
    const int half = p.R / 2;
    const uint16_t* cs = p.cos + row * p.R;
    const uint16_t* sn = p.sin + row * p.R;
    in.c1 = __ldcs(reinterpret_cast<const uint2*>(cs + 4 * lane));
    in.c2 = __ldcs(reinterpret_cast<const uint2*>(cs + half + 4 * lane));
    in.s1 = __ldcs(reinterpret_cast<const uint2*>(sn + 4 * lane));
    in.s2 = __ldcs(reinterpret_cast<const uint2*>(sn + half + 4 * lane));
  }
  const int64_t s = row % p.S;
  const int64_t b = row / (p.S * p.N);
  in.slot = __ldg(p.index + b * p.S + s);
}

template <int VARIANT, bool QK, bool QV, int CPL>
__global__ void __launch_bounds__(kThreads) kv_rms_norm_rope_cache_kernel(const KvLaunch p) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = p.B * p.N * p.S;
  const int R = p.R, half = R / 2, rope_lanes = R / 8;
  const int rms = VARIANT == 1 ? static_cast<int>(p.Dkv) - R : static_cast<int>(p.Dkv);
  const int rms_chunks = rms / 8;
  const int kw = VARIANT == 1 ? R : static_cast<int>(p.Dkv);
  const int cw = VARIANT == 1 ? rms : static_cast<int>(p.Dv);
  const int v_chunks = VARIANT == 2 ? cw / 8 : 0;
  const int64_t slots = p.block_num * p.block_size;
  const size_t k_elt = QK ? 1 : 2, c_elt = QV ? 1 : 2;

  // gamma is the same for every row: keep the lane's chunks in registers
  uint4 gam[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = lane + 32 * i;
    gam[i] = c < rms_chunks ? __ldg(reinterpret_cast<const uint4*>(p.gamma + 8 * c))
                            : make_uint4(0, 0, 0, 0);
  }

  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
  int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  RowIn<CPL> cur;
  if (row < rows) load_row<VARIANT, CPL>(p, row, lane, rms, rms_chunks, v_chunks, rope_lanes, cur);

  while (row < rows) {
    const int64_t next = row + stride;
    RowIn<CPL> nxt;
    if (next < rows) load_row<VARIANT, CPL>(p, next, lane, rms, rms_chunks, v_chunks, rope_lanes, nxt);

    const int n = static_cast<int>((row / p.S) % p.N);

    // (1) RmsNorm
    float y[CPL][8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      unpack8(cur.x[i], y[i]);
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(y[i][j], y[i][j], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss / static_cast<float>(rms) + p.eps);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      float g[8];
      unpack8(gam[i], g);
#pragma unroll
      for (int j = 0; j < 8; ++j) y[i][j] = y[i][j] * inv * g[j];
    }

    // (4) slot of this token
    const int64_t slot = cur.slot;
    const bool to_cache = slot >= 0 && slot < slots;
    if (!to_cache && slot != -1 && n == 0 && lane == 0 && p.err_count != nullptr)
      atomicAdd(p.err_count, 1);  // once per token, not per head
    const int64_t blk = to_cache ? slot / p.block_size : 0;
    const int64_t off = to_cache ? slot % p.block_size : 0;
    const int64_t cache_row = p.mode == 2 ? (blk * p.N + n) * p.block_size + off
                                          : (blk * p.block_size + off) * p.N + n;
    void* k_row = static_cast<uint8_t*>(p.k_cache) + static_cast<size_t>(cache_row) * kw * k_elt;
    void* c_row = static_cast<uint8_t*>(p.ckv_cache) + static_cast<size_t>(cache_row) * cw * c_elt;
    const float* ksc = QK ? p.k_scale + (VARIANT == 2 ? n * kw : 0) : nullptr;
    const float* kof = (QK && p.k_offset) ? p.k_offset + (VARIANT == 2 ? n * kw : 0) : nullptr;
    const float* vsc = QV ? p.v_scale + (VARIANT == 2 ? n * cw : 0) : nullptr;
    const float* vof = (QV && p.v_offset) ? p.v_offset + (VARIANT == 2 ? n * cw : 0) : nullptr;
    uint16_t* kr_row = p.out_kv ? p.k_rope + row * kw : nullptr;
    uint16_t* ckv_row = p.out_kv ? p.c_kv + row * cw : nullptr;

    // (2) interleaved RoPE: lane l owns pairs j = 4l .. 4l+3
    if (lane < rope_lanes) {
      float r[8];
      if (VARIANT == 1) {
        unpack8(cur.xr, r);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = y[0][j];
      }
      const float cc1[4] = {bf16_lo(cur.c1.x), bf16_hi(cur.c1.x), bf16_lo(cur.c1.y), bf16_hi(cur.c1.y)};
      const float cc2[4] = {bf16_lo(cur.c2.x), bf16_hi(cur.c2.x), bf16_lo(cur.c2.y), bf16_hi(cur.c2.y)};
      const float ss1[4] = {bf16_lo(cur.s1.x), bf16_hi(cur.s1.x), bf16_lo(cur.s1.y), bf16_hi(cur.s1.y)};
      const float ss2[4] = {bf16_lo(cur.s2.x), bf16_hi(cur.s2.x), bf16_lo(cur.s2.y), bf16_hi(cur.s2.y)};
      float o1[4], o2[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float x1 = r[2 * m], x2 = r[2 * m + 1];
        o1[m] = x1 * cc1[m] - x2 * ss1[m];
        o2[m] = x2 * cc2[m] + x1 * ss2[m];
      }
      if (to_cache) {
        store_vals<QK, 4>(k_row, 4 * lane, o1, ksc, kof);
        store_vals<QK, 4>(k_row, half + 4 * lane, o2, ksc, kof);
      }
      if (kr_row != nullptr) {
        store_vals<false, 4>(kr_row, 4 * lane, o1, nullptr, nullptr);
        store_vals<false, 4>(kr_row, half + 4 * lane, o2, nullptr, nullptr);
      }
    }

    if (VARIANT == 2) {
      // rope_out tail = y[..., rope_size:]
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c >= rope_lanes && c < rms_chunks) {
          if (to_cache) store_vals<QK, 8>(k_row, 8 * c, y[i], ksc, kof);
          if (kr_row != nullptr) store_vals<false, 8>(kr_row, 8 * c, y[i], nullptr, nullptr);
        }
      }
      // ckv <- v_optional
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < v_chunks) {
          if (to_cache) {
            if constexpr (QV) {
              float f[8];
              unpack8(cur.v[i], f);
              store_vals<true, 8>(c_row, 8 * c, f, vsc, vof);
            } else {
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(c_row) + 8 * c) = cur.v[i];
            }
          }
          if (ckv_row != nullptr) *reinterpret_cast<uint4*>(ckv_row + 8 * c) = cur.v[i];
        }
      }
    } else {
      // ckv <- y
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < rms_chunks) {
          if (to_cache) store_vals<QV, 8>(c_row, 8 * c, y[i], vsc, vof);
          if (ckv_row != nullptr) store_vals<false, 8>(ckv_row, 8 * c, y[i], nullptr, nullptr);
        }
      }
    }
    cur = nxt;
    row = next;
  }
}

// persistent grid: as many blocks as fit on the GPU at once, capped by the row count
template <typename K>
unsigned persistent_grid(K kernel, int64_t rows) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (rows + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(per_sm) * device_sm_count();
  return static_cast<unsigned>(want < cap ? want : cap);
}

template <int VARIANT, bool QK, bool QV, int CPL>
cudaError_t launch_one(const KvLaunch& L, cudaStream_t st) {
  auto kernel = kv_rms_norm_rope_cache_kernel<VARIANT, QK, QV, CPL>;
  const unsigned grid = persistent_grid(kernel, L.B * L.N * L.S);
  kernel<<<grid, kThreads, 0, st>>>(L);
  return cudaGetLastError();
}

template <int VARIANT, bool QK, bool QV>
cudaError_t launch_cpl(const KvLaunch& L, int cpl, unsigned, cudaStream_t st) {
  switch (cpl) {
    case 1: return launch_one<VARIANT, QK, QV, 1>(L, st);
    case 2: return launch_one<VARIANT, QK, QV, 2>(L, st);
    case 4: return launch_one<VARIANT, QK, QV, 4>(L, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int VARIANT>
cudaError_t launch_variant(const KvLaunch& L, int cpl, unsigned grid, cudaStream_t st) {
  const bool qk = L.k_scale != nullptr, qv = L.v_scale != nullptr;
  if (qk && qv) return launch_cpl<VARIANT, true, true>(L, cpl, grid, st);
  if (qk) return launch_cpl<VARIANT, true, false>(L, cpl, grid, st);
  if (qv) return launch_cpl<VARIANT, false, true>(L, cpl, grid, st);
  return launch_cpl<VARIANT, false, false>(L, cpl, grid, st);
}

}  // namespace

cudaError_t launch_kv_rms_norm_rope_cache(const KvLaunch& L, cudaStream_t stream) {
  const int64_t rms = L.variant == 1 ? L.Dkv - L.R : L.Dkv;
  int64_t chunks = rms / 8;
  if (L.variant == 2 && L.Dv / 8 > chunks) chunks = L.Dv / 8;  // v_optional rides the same lanes
  const int cpl = chunks <= 32 ? 1 : (chunks <= 64 ? 2 : 4);
  if (chunks > 128) return cudaErrorInvalidValue;
  const unsigned grid = 0;
  return L.variant == 1 ? launch_variant<1>(L, cpl, grid, stream)
                        : launch_variant<2>(L, cpl, grid, stream);
}

}  // namespace ra
