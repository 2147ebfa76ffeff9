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
// GB300 mapping: an HBM stream of short rows (0.6-1.4 KB).  The two row shapes
// of the common calls (V1 576 = 512 + 64, V2 192 / 128 with RoPE on 64) in the
// paged modes with int8 or 16-bit caches run the bulk-copy pipelined kernel
// further down; every other call runs this register kernel, built to keep bytes
// in flight with few instructions per byte:
//  * persistent warps, each owning a contiguous range of (b, n, s) rows and
//    walking (b, n, s) incrementally (no integer division per row);
//  * a warp works on 32 / LPR rows at once, LPR = 8, 16 or 32 lanes per row
//    (the fewest that hold the RoPE pairs with at most four 16-byte chunks per
//    lane), so every lane has work in every phase and per-row costs (slot
//    lookup, addressing, the RMS shuffle tree) are shared;
//  * two row groups in registers per lane: one is processed while the next loads;
//  * the per-channel quantisation scales and offsets (per head in V2) are
//    staged once per block in shared memory, laid out for conflict-free reads;
//  * packed fp32x2 arithmetic; int8 codes are rounded with cvt.rni and packed
//    with saturation by cvt.pack.sat;
//  * lane j < rope_size/8 of a row owns interleaved pairs 4j..4j+3, whose outputs
//    land at positions 4j and rope_size/2 + 4j of the de-interleaved result.
//    Cache rows are contiguous, so each scattered slot is written with whole vectors.
#include <cuda_fp8.h>

#include <atomic>

#include "internal.h"
#include "kv_cache.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

// 16-bit input elements: bf16 or fp16 (F16), two per 32-bit word, first in the low half
template <bool F16>
__device__ __forceinline__ float2 to_f2(uint32_t w) {
  if constexpr (F16) return __half22float2(*reinterpret_cast<const __half2*>(&w));
  else return make_float2(bf16_lo(w), bf16_hi(w));
}
template <bool F16>
__device__ __forceinline__ uint32_t from_f2(float a, float b) {
  if constexpr (F16) return pack_f16x2(a, b);
  else return pack_bf16x2(a, b);
}
template <bool F16>
__device__ __forceinline__ void unpack8(uint4 u, float2 (&f)[4]) {
  f[0] = to_f2<F16>(u.x);
  f[1] = to_f2<F16>(u.y);
  f[2] = to_f2<F16>(u.z);
  f[3] = to_f2<F16>(u.w);
}
template <bool F16>
__device__ __forceinline__ uint4 pack8(const float2 (&f)[4]) {
  uint4 u;
  u.x = from_f2<F16>(f[0].x, f[0].y);
  u.y = from_f2<F16>(f[1].x, f[1].y);
  u.z = from_f2<F16>(f[2].x, f[2].y);
  u.w = from_f2<F16>(f[3].x, f[3].y);
  return u;
}
// four quantised codes of v * scale + offset (one fp32 rounding), the first channel
// in the lowest byte.  int8 (formula (3)): round half to even, saturated to
// [-128, 127] -- cvt.rni saturates at the int32 range and cvt.pack.sat (PTX ISA,
// sm_72+) clamps each value to the int8 range as it packs two of them above the
// 16 bits taken from its third operand.  FP8: the hardware E4M3 / E5M2 conversion,
// round to nearest even, saturated at the largest finite value.
template <bool GEN>
__device__ __forceinline__ uint32_t quant4(float2 v01, float2 v23, float4 sc, float4 of, int32_t qt) {
  const float a = fmaf(v01.x, sc.x, of.x), b = fmaf(v01.y, sc.y, of.y);
  const float c = fmaf(v23.x, sc.z, of.z), d = fmaf(v23.y, sc.w, of.w);
  if (!GEN || qt == kQuantInt8) {
    uint32_t hi, r;
    asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi) : "r"(__float2int_rn(d)), "r"(__float2int_rn(c)));
    asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(__float2int_rn(b)), "r"(__float2int_rn(a)), "r"(hi));
    return r;
  }
  const __nv_fp8_interpretation_t k = qt == kQuantE4m3 ? __NV_E4M3 : __NV_E5M2;
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, k);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, k);
  return lo | (hi << 16);
}

// Quantisation tables in shared memory, in units of 4 channels (a float4 of
// scales, and one of offsets, for channels 4u..4u+3), heads one after another
// `stride` apart.  Within a head, group u sits at (u odd ? odd : 0) + (u / 2) * step.
//  * split layout (step 1, odd = 4 mod 8): a lane that quantises the 8 channels of
//    chunk c reads positions c and odd + c, one that quantises 4 reads u / 2 or
//    odd + u / 2, so with the lanes of a quarter warp on consecutive chunks (or
//    groups) their 16-byte reads land in distinct banks;
//  * plain layout (step 2, odd 1): group u at u; chunk c reads 2c and 2c + 1, two
//    lanes of a quarter warp per bank.
struct TabLayout {
  int odd, step, stride;  // float4 units
};
__host__ __device__ inline TabLayout tab_layout(int width, bool split) {  // width % 8 == 0
  if (!split) return TabLayout{1, 2, width / 4};
  const int half = width / 8;  // groups of each parity
  const int odd = half + (12 - half % 8) % 8;
  return TabLayout{odd, 1, odd + half};
}
struct QuantTab {
  const float4* scale;
  const float4* offset;
  int odd, step, stride;
};
// Fills one table (every head) from the per-channel scale / offset arrays, or
// from their one value when they are [1] (`scalar`).
__device__ __forceinline__ void fill_table(float4* ts, float4* to, const float* scale, const float* offset,
                                           int heads, int width, TabLayout l, bool scalar,
                                           int tid, int nthreads) {
  const int groups = width / 4, n = heads * groups;
  for (int e = tid; e < n; e += nthreads) {
    const int hd = e / groups, u = e - hd * groups;
    const int pos = hd * l.stride + ((u & 1) ? l.odd : 0) + (u >> 1) * l.step;
    if (scalar) {
      const float s0 = __ldg(scale), o0 = offset ? __ldg(offset) : 0.f;
      ts[pos] = make_float4(s0, s0, s0, s0);
      to[pos] = make_float4(o0, o0, o0, o0);
    } else {
      ts[pos] = __ldg(reinterpret_cast<const float4*>(scale) + e);
      to[pos] = offset ? __ldg(reinterpret_cast<const float4*>(offset) + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// 8 channels starting at `ch` (a multiple of 8) of a cache row: quantised (qt != 0,
// one byte each) or in the input dtype
template <bool F16, bool GEN>
__device__ __forceinline__ void store8(int32_t qt, void* row_base, int ch, const float2 (&v)[4],
                                       QuantTab t) {
  if (qt != kQuantNone) {
    const int c = ch >> 3;
    uint2 w;
    const int e = c * t.step;
    w.x = quant4<GEN>(v[0], v[1], t.scale[e], t.offset[e], qt);
    w.y = quant4<GEN>(v[2], v[3], t.scale[t.odd + e], t.offset[t.odd + e], qt);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(row_base) + ch) = w;
  } else {
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(row_base) + ch) = pack8<F16>(v);
  }
}
// 4 channels starting at `ch` (a multiple of 4)
template <bool F16, bool GEN>
__device__ __forceinline__ void store4(int32_t qt, void* row_base, int ch, float2 v01, float2 v23,
                                       QuantTab t) {
  if (qt != kQuantNone) {
    const int u = ch >> 2, pos = ((u & 1) ? t.odd : 0) + (u >> 1) * t.step;
    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(row_base) + ch) =
        quant4<GEN>(v01, v23, t.scale[pos], t.offset[pos], qt);
  } else {
    uint2 w;
    w.x = from_f2<F16>(v01.x, v01.y);
    w.y = from_f2<F16>(v23.x, v23.y);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(row_base) + ch) = w;
  }
}

// The row shapes of the pipelined kernel, compiled in so that the per-row
// addressing and the chunk tests fold to constants.
template <int SHAPE>
struct RowShape;
template <>
struct RowShape<1> {  // V1, the MLA combined kv: 512 normed + 64 RoPE channels
  static constexpr int dkv = 576, dv = 512, r = 64;
};
template <>
struct RowShape<2> {  // V2: kv of 192 channels (RoPE on the first 64), v of 128
  static constexpr int dkv = 192, dv = 128, r = 64;
};

// Launch constants computed on the host.
struct KvAux {
  float inv_rms;      // 1 / rms_size
  int32_t bs_shift;   // log2(block_size) when it is a power of two, else -1
  int32_t blocks_per_batch;  // PA_BLK_BNSD: ceil(S / block_size) index entries per batch
};

// What one lane needs from HBM for its row of a row group, as raw vectors, so
// that the next group's loads are in flight while this one is processed.
template <int CPL>
struct RowIn {
  uint4 x[CPL];            // kv chunks j + LPR*i of the RMSNorm part
  uint4 xr;                // V1: chunk j of the raw RoPE part
  uint4 v[CPL];            // V2: chunks j + LPR*i of v_optional
  uint2 c1, c2, s1, s2;    // cos/sin of pairs 4j..4j+3, at j and R/2 + j
  int64_t slot;            // the index entry (PA_BLK_BNSD: the start of the token's block)
  int32_t n;
  int32_t aux;             // Norm: the batch b; PA_BLK_BNSD: s % block_size
};

// (b, n, s) of one row, advanced without division.
struct Cursor {
  int64_t row, tok;        // tok = b * S + s
  int32_t b, n, s;
  __device__ __forceinline__ void advance(int32_t step, int32_t N, int32_t S) {
    row += step;
    tok += step;
    s += step;
    while (s >= S) {
      s -= S;
      tok -= S;
      if (++n == N) {
        n = 0;
        ++b;
        tok += S;
      }
    }
  }
};

// GEN: the general kernel (Norm and PA_BLK_BNSD modes, S-broadcast cos/sin, FP8
// caches); without it only PA / PA_BNSD with int8 or 16-bit caches is compiled in.
// JLO: lane = g * LPR + j (a row's lanes adjacent), else lane = j * (32 / LPR) + g.
template <int VARIANT, int LPR, int CPL, bool F16, bool GEN, bool JLO = false>
struct KvRows {
  const KvLaunch& p;
  KvAux aux;
  int j;
  int dkv, dv, r;
  int rms, rms_chunks, v_chunks, rope_lanes, half, kw, cw;
  int64_t slots;
  const uint4 (&gam)[CPL];
  QuantTab kt0, vt0;

  __device__ __forceinline__ void load(const Cursor& c, bool valid, RowIn<CPL>& in) const {
    const uint4 z = make_uint4(0, 0, 0, 0);
    const uint16_t* x = p.kv + c.row * dkv;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int ch = j + LPR * i;
      in.x[i] = valid && ch < rms_chunks ? __ldcs(reinterpret_cast<const uint4*>(x + 8 * ch)) : z;
    }
    if (VARIANT == 1)
      in.xr = valid && j < rope_lanes ? __ldcs(reinterpret_cast<const uint4*>(x + rms + 8 * j)) : z;
    if (VARIANT == 2) {
      const uint16_t* vrow = p.v + c.row * dv;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int ch = j + LPR * i;
        in.v[i] = valid && ch < v_chunks ? __ldcs(reinterpret_cast<const uint4*>(vrow + 8 * ch)) : z;
      }
    }
    if (valid && j < rope_lanes) {
      // cos/sin row: (b, n, s), or (b, n, 0) when they are broadcast over S
      const int64_t rrow = GEN && p.rope_bcast ? static_cast<int64_t>(c.b) * p.N + c.n : c.row;
      const uint16_t* cs = p.cos + rrow * r;
      const uint16_t* sn = p.sin + rrow * r;
      in.c1 = __ldcs(reinterpret_cast<const uint2*>(cs + 4 * j));
      in.c2 = __ldcs(reinterpret_cast<const uint2*>(cs + half + 4 * j));
      in.s1 = __ldcs(reinterpret_cast<const uint2*>(sn + 4 * j));
      in.s2 = __ldcs(reinterpret_cast<const uint2*>(sn + half + 4 * j));
    }
    // the index entry of this token (PA_BLK_BNSD: of its block of block_size tokens)
    int64_t ipos = c.tok;
    in.aux = GEN && p.mode == kModeNorm ? c.b : 0;
    if (GEN && p.mode == kModePaBlkBnsd) {
      const int32_t blk = aux.bs_shift >= 0 ? c.s >> aux.bs_shift : static_cast<int32_t>(c.s / p.block_size);
      ipos = static_cast<int64_t>(c.b) * aux.blocks_per_batch + blk;
      in.aux = c.s - static_cast<int32_t>(static_cast<int64_t>(blk) * p.block_size);
    }
    in.slot = valid ? __ldg(p.index + ipos) : int64_t(-1);
    in.n = c.n;
  }

  __device__ __forceinline__ void process(const RowIn<CPL>& in, int64_t row, bool valid) const {
    const int n = in.n;
    // (1) RmsNorm over the row's LPR lanes
    float2 y[CPL][4];
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      unpack8<F16>(in.x[i], y[i]);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc = __ffma2_rn(y[i][k], y[i][k], acc);
    }
    float ss = acc.x + acc.y;
    if constexpr (JLO) {
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    } else {
#pragma unroll
      for (int o = 16; o >= 32 / LPR; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    }
    const float inv = rsqrtf(fmaf(ss, aux.inv_rms, p.eps));
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      float2 g[4];
      unpack8<F16>(gam[i], g);
#pragma unroll
      for (int k = 0; k < 4; ++k) y[i][k] = __fmul2_rn(__fmul2_rn(y[i][k], inv2), g[k]);
    }
    if (!valid) return;

    // (4) slot of this token: the index entry, in PA_BLK_BNSD plus the token's place in its block
    int64_t slot = in.slot;
    if (GEN && p.mode == kModePaBlkBnsd && slot >= 0) slot += in.aux;
    const bool to_cache = slot >= 0 && slot < slots;
    if (!to_cache && slot != -1 && n == 0 && j == 0 && p.err_count != nullptr)
      atomicAdd(p.err_count, 1);  // once per token, not per head
    int64_t cache_row = 0;
    if (to_cache) {
      if (GEN && p.mode == kModeNorm) {  // [B, N, Scache, D]
        cache_row = (static_cast<int64_t>(in.aux) * p.N + n) * p.cache_seq + slot;
      } else {
        int64_t blk, off;
        if (aux.bs_shift >= 0) {
          blk = slot >> aux.bs_shift;
          off = slot & (p.block_size - 1);
        } else {
          blk = slot / p.block_size;
          off = slot - blk * p.block_size;
        }
        cache_row = p.mode == kModePa ? (blk * p.block_size + off) * p.N + n   // [bn, bs, N, D]
                                      : (blk * p.N + n) * p.block_size + off;  // [bn, N, bs, D]
      }
    }
    const int32_t qk = p.kq, qv = p.vq;
    void* k_row = static_cast<uint8_t*>(p.k_cache) + static_cast<size_t>(cache_row) * kw * (qk ? 1 : 2);
    void* c_row = static_cast<uint8_t*>(p.ckv_cache) + static_cast<size_t>(cache_row) * cw * (qv ? 1 : 2);
    const int kh = VARIANT == 2 ? n * kt0.stride : 0, vh = VARIANT == 2 ? n * vt0.stride : 0;
    const QuantTab kt{kt0.scale + kh, kt0.offset + kh, kt0.odd, kt0.step, kt0.stride};
    const QuantTab vt{vt0.scale + vh, vt0.offset + vh, vt0.odd, vt0.step, vt0.stride};
    uint16_t* kr_row = p.out_kv ? p.k_rope + row * kw : nullptr;
    uint16_t* ckv_row = p.out_kv ? p.c_kv + row * cw : nullptr;

    // (2) interleaved RoPE: lane j owns pairs 4j .. 4j+3
    if (j < rope_lanes) {
      float2 r[4];
      if (VARIANT == 1) {
        unpack8<F16>(in.xr, r);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = y[0][k];
      }
      // r[m] = (x1, x2) of pair 4j + m
      const float2 c1a = to_f2<F16>(in.c1.x), c1b = to_f2<F16>(in.c1.y);
      const float2 c2a = to_f2<F16>(in.c2.x), c2b = to_f2<F16>(in.c2.y);
      const float2 s1a = to_f2<F16>(in.s1.x), s1b = to_f2<F16>(in.s1.y);
      const float2 s2a = to_f2<F16>(in.s2.x), s2b = to_f2<F16>(in.s2.y);
      const float2 x1a = make_float2(r[0].x, r[1].x), x1b = make_float2(r[2].x, r[3].x);
      const float2 x2a = make_float2(r[0].y, r[1].y), x2b = make_float2(r[2].y, r[3].y);
      // out_m = x1 cos_m - x2 sin_m ; out_{R/2+m} = x2 cos_{R/2+m} + x1 sin_{R/2+m}
      const float2 o1a = __ffma2_rn(x1a, c1a, __fmul2_rn(x2a, make_float2(-s1a.x, -s1a.y)));
      const float2 o1b = __ffma2_rn(x1b, c1b, __fmul2_rn(x2b, make_float2(-s1b.x, -s1b.y)));
      const float2 o2a = __ffma2_rn(x2a, c2a, __fmul2_rn(x1a, s2a));
      const float2 o2b = __ffma2_rn(x2b, c2b, __fmul2_rn(x1b, s2b));
      if (to_cache) {
        store4<F16, GEN>(qk, k_row, 4 * j, o1a, o1b, kt);
        store4<F16, GEN>(qk, k_row, half + 4 * j, o2a, o2b, kt);
      }
      if (kr_row != nullptr) {
        store4<F16, GEN>(kQuantNone, kr_row, 4 * j, o1a, o1b, kt);
        store4<F16, GEN>(kQuantNone, kr_row, half + 4 * j, o2a, o2b, kt);
      }
    }

    if (VARIANT == 2) {
      // rope_out tail = y[..., rope_size:]
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int ch = j + LPR * i;
        if (ch >= rope_lanes && ch < rms_chunks) {
          if (to_cache) store8<F16, GEN>(qk, k_row, 8 * ch, y[i], kt);
          if (kr_row != nullptr) store8<F16, GEN>(kQuantNone, kr_row, 8 * ch, y[i], kt);
        }
      }
      // ckv <- v_optional
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int ch = j + LPR * i;
        if (ch < v_chunks) {
          if (to_cache) {
            if (qv) {
              float2 f[4];
              unpack8<F16>(in.v[i], f);
              store8<F16, GEN>(qv, c_row, 8 * ch, f, vt);
            } else {
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(c_row) + 8 * ch) = in.v[i];
            }
          }
          if (ckv_row != nullptr) *reinterpret_cast<uint4*>(ckv_row + 8 * ch) = in.v[i];
        }
      }
    } else {
      // ckv <- y
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int ch = j + LPR * i;
        if (ch < rms_chunks) {
          if (to_cache) store8<F16, GEN>(qv, c_row, 8 * ch, y[i], vt);
          if (ckv_row != nullptr) store8<F16, GEN>(kQuantNone, ckv_row, 8 * ch, y[i], vt);
        }
      }
    }
  }
};

// Shared-memory bytes of the quantisation tables (scale and offset, per head in V2).
size_t quant_table_bytes(const KvLaunch& L, bool qk, bool qv, bool split) {
  const int64_t heads = L.variant == 2 ? L.N : 1;
  const int kw = static_cast<int>(L.variant == 1 ? L.R : L.Dkv);
  const int cw = static_cast<int>(L.variant == 1 ? L.Dkv - L.R : L.Dv);
  const int64_t units = (qk ? tab_layout(kw, split).stride : 0) + (qv ? tab_layout(cw, split).stride : 0);
  return static_cast<size_t>(heads * units) * 2 * sizeof(float4);
}

constexpr int kMinBlocks = 3;  // 12 warps per SM: up to 168 registers per thread

template <int VARIANT, int LPR, int CPL, bool F16, bool GEN>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    kv_rms_norm_rope_cache_kernel(const KvLaunch p, const KvAux aux) {
  extern __shared__ float4 tabs[];
  constexpr int DEPTH = 2;          // row-group buffers per lane: one processed, one loading
  constexpr int RPG = 32 / LPR;     // rows per warp per step
  const int lane = threadIdx.x & 31;
  const int g = lane % RPG, j = lane / RPG;
  const int64_t rows = p.B * p.N * p.S;
  const int R = p.R;
  const int dkv = static_cast<int>(p.Dkv), dv = static_cast<int>(p.Dv);
  const int rms = VARIANT == 1 ? dkv - R : dkv;
  const int kw = VARIANT == 1 ? R : dkv;
  const int cw = VARIANT == 1 ? rms : dv;
  const int heads = VARIANT == 2 ? static_cast<int>(p.N) : 1;
  const int32_t N = static_cast<int32_t>(p.N), S = static_cast<int32_t>(p.S);

  // this warp's contiguous range of rows, a multiple of RPG long
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t per_warp = ((rows + warps - 1) / warps + RPG - 1) / RPG * RPG;
  const int64_t r_begin = (static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * per_warp;
  const int64_t r_end = r_begin + per_warp < rows ? r_begin + per_warp : rows;

  uint4 gam[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int ch = j + LPR * i;
    gam[i] = ch * 8 < rms ? __ldg(reinterpret_cast<const uint4*>(p.gamma + 8 * ch)) : make_uint4(0, 0, 0, 0);
  }
  const TabLayout kl = tab_layout(kw, true), vl = tab_layout(cw, true);
  const int ku = p.kq ? heads * kl.stride : 0, vu = p.vq ? heads * vl.stride : 0;
  float4* ks = tabs;
  float4* ko = ks + ku;
  float4* vs = ko + ku;
  float4* vo = vs + vu;
  const int64_t slots = p.mode == kModeNorm ? p.cache_seq : p.block_num * p.block_size;
  const KvRows<VARIANT, LPR, CPL, F16, GEN> w{p, aux, j, dkv, dv, R, rms, rms / 8, VARIANT == 2 ? cw / 8 : 0, R / 8, R / 2, kw, cw,
                                         slots, gam, QuantTab{ks, ko, kl.odd, kl.step, kl.stride},
                                         QuantTab{vs, vo, vl.odd, vl.step, vl.stride}};

  // the lane's load cursor: row r_begin + g, then RPG rows further each step
  Cursor cur;
  {
    int64_t start = r_begin + g;
    if (start >= rows) start = 0;
    const int64_t per_b = p.N * p.S;
    const int64_t b = start / per_b, rem = start - b * per_b;
    cur.row = start;
    cur.b = static_cast<int32_t>(b);
    cur.n = static_cast<int32_t>(rem / p.S);
    cur.s = static_cast<int32_t>(rem - static_cast<int64_t>(cur.n) * p.S);
    cur.tok = b * p.S + cur.s;
    if (r_begin + g >= rows) cur.row = r_begin + g;  // never valid
  }
  // start the first groups' loads before staging the tables
  RowIn<CPL> buf[DEPTH];
  int64_t next = r_begin;  // first row of the next group to load (warp-uniform)
#pragma unroll
  for (int k = 0; k < DEPTH; ++k) {
    if (next < r_end) {
      w.load(cur, cur.row < r_end, buf[k]);
      cur.advance(RPG, N, S);
      next += RPG;
    }
  }
  if (p.kq) fill_table(ks, ko, p.k_scale, p.k_offset, heads, kw, kl, p.k_scalar != 0, threadIdx.x, blockDim.x);
  if (p.vq) fill_table(vs, vo, p.v_scale, p.v_offset, heads, cw, vl, p.v_scalar != 0, threadIdx.x, blockDim.x);
  __syncthreads();

  for (int64_t base = r_begin; base < r_end; base += DEPTH * RPG) {
#pragma unroll
    for (int k = 0; k < DEPTH; ++k) {
      const int64_t grp = base + k * RPG;
      if (grp < r_end) {
        w.process(buf[k], grp + g, grp + g < r_end);
        if (next < r_end) {
          w.load(cur, cur.row < r_end, buf[k]);
          cur.advance(RPG, N, S);
          next += RPG;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- staged kernel
// For the two common row shapes, in every cache mode and cache type.  A tile of
// consecutive (b, n, s) rows is one contiguous span in each of kv, v,
// cos and sin, so one lane of a producer warp moves it into shared memory with
// four bulk copies (cp.async.bulk, completion counted by the stage's mbarrier;
// with S-broadcast cos/sin only kv and v are copied, and the consumers read the
// one cos/sin row of each (b, n), which stays cached, straight from global memory),
// kStages - 1 tiles ahead of the consumer warps.  The producer warp also looks up
// each row's head, its index entry (per token, or per block of block_size tokens
// in PA_BLK_BNSD) and the row's batch (Norm) or place in its block (PA_BLK_BNSD).  The consumers run the same row arithmetic as
// the kernel above on operands read from shared memory, with a row's lanes
// adjacent so that those reads are free of bank conflicts.  Every wait has a time
// limit: when one runs out the block records it in the status word and leaves,
// the producer first waiting (with a limit) for the copies it issued.
constexpr int kStages = 3;

__device__ int32_t g_kv_status;

// Shared-memory plan of the staged kernel, in bytes from the dynamic base.
struct StagedPlan {
  uint32_t tables, stage_bytes, stages, slots, heads, auxs, bns, bars, flag, total;
};
__host__ __device__ inline StagedPlan staged_plan(uint32_t table_bytes, uint32_t stage_bytes, uint32_t tile_rows) {
  StagedPlan pl;
  pl.tables = 0;
  pl.stage_bytes = stage_bytes;
  pl.stages = (table_bytes + 127u) & ~127u;
  pl.slots = pl.stages + kStages * stage_bytes;
  pl.heads = pl.slots + kStages * tile_rows * 8;
  pl.auxs = pl.heads + kStages * tile_rows * 4;
  pl.bns = pl.auxs + kStages * tile_rows * 4;
  pl.bars = pl.bns + kStages * tile_rows * 4;
  pl.flag = pl.bars + 2 * kStages * 8;
  pl.total = pl.flag + 16;
  return pl;
}

template <int VARIANT>
struct StagedShape {
  using Sh = RowShape<VARIANT>;
  static constexpr int R = Sh::r, DKV = Sh::dkv, DV = VARIANT == 2 ? Sh::dv : 0;
  static constexpr int RMS = VARIANT == 1 ? DKV - R : DKV;
  static constexpr int KW = VARIANT == 1 ? R : DKV, CW = VARIANT == 1 ? RMS : Sh::dv;
  static constexpr int LPR = VARIANT == 1 ? 16 : 8, CPL = VARIANT == 1 ? 4 : 3, RPG = 32 / LPR;
  // tile rows, consumer warps and blocks per SM.  V2 rows (640 B) take tiles of 32 rows
  // for 8 consumer warps, two blocks per SM: 0.0525 ms at 720p against 0.0543 ms for
  // 16-row tiles, 4 warps and three blocks (S-broadcast: 0.0537 against 0.0584).  V1
  // rows (1408 B) keep 16-row tiles: with 32 they fit one block per SM and took
  // 0.080 ms against 0.073 ms (int8 MLA call)
  static constexpr int TILE = VARIANT == 1 ? 16 : 32, CWARPS = VARIANT == 1 ? 4 : 8;
  static constexpr int THREADS = (CWARPS + 1) * 32, MIN_BLOCKS = VARIANT == 1 ? 3 : 2;
  static constexpr uint32_t KV_B = TILE * DKV * 2, V_B = TILE * DV * 2, CS_B = TILE * R * 2;
  static constexpr uint32_t STAGE_B = KV_B + V_B + 2 * CS_B;
  static constexpr uint32_t ROW_B = STAGE_B / TILE;
  static constexpr int STEPS = TILE / (CWARPS * RPG);  // row groups per consumer warp and tile
  // V1 keeps the plain table layout: its step (a DRAM-bound mix of reads and
  // row-contiguous output writes) measured faster with it (74 vs 77 us), though
  // the split layout has fewer bank conflicts.
  static constexpr bool SPLIT = VARIANT == 2;
  static_assert(STEPS * CWARPS * RPG == TILE, "tile rows split evenly over the consumer warps");
  static_assert(TILE <= 32, "one producer lane per tile row");
  static_assert(RMS / 8 <= LPR * CPL && Sh::dv / 8 <= LPR * CPL && R / 8 <= LPR, "lane layout holds the row");
};

// GEN: Norm / PA_BLK_BNSD addressing and FP8 caches compiled in
template <int VARIANT, bool F16, bool GEN>
__global__ void __launch_bounds__(StagedShape<VARIANT>::THREADS, StagedShape<VARIANT>::MIN_BLOCKS)
    kv_staged_kernel(const KvLaunch p, const KvAux aux, const uint32_t tiles) {
  using T = StagedShape<VARIANT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rows = static_cast<uint32_t>(p.B * p.N * p.S);
  const uint32_t S = static_cast<uint32_t>(p.S), N = static_cast<uint32_t>(p.N);
  const int heads = VARIANT == 2 ? static_cast<int>(p.N) : 1;
  const TabLayout kl = tab_layout(T::KW, T::SPLIT), vl = tab_layout(T::CW, T::SPLIT);
  const int ku = p.kq ? heads * kl.stride : 0, vu = p.vq ? heads * vl.stride : 0;
  const StagedPlan pl = staged_plan(static_cast<uint32_t>(2 * (ku + vu) * 16), T::STAGE_B, T::TILE);
  float4* ks = reinterpret_cast<float4*>(smem);
  float4* ko = ks + ku;
  float4* vs = ko + ku;
  float4* vo = vs + vu;
  int64_t* slot_s = reinterpret_cast<int64_t*>(smem + pl.slots);
  int32_t* head_s = reinterpret_cast<int32_t*>(smem + pl.heads);
  int32_t* aux_s = reinterpret_cast<int32_t*>(smem + pl.auxs);
  int32_t* bn_s = reinterpret_cast<int32_t*>(smem + pl.bns);  // b * N + n (S-broadcast cos/sin row)
  const bool bcast = GEN && p.rope_bcast;
  const uint32_t bars = smem_u32(smem + pl.bars);  // full[kStages], then empty[kStages]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + pl.flag);
  const uint32_t stage0 = smem_u32(smem + pl.stages);
  const uint64_t limit = static_cast<uint64_t>(p.wait_ns);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars + 8 * s, 32);                           // every producer lane arrives
      mbar_init(bars + 8 * (kStages + s), T::CWARPS);   // one arrive per consumer warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == T::CWARPS) {
    // producer: tile k of this block goes to stage k % kStages
    uint32_t k = 0;
    bool live = true;
    for (uint32_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++k) {
      const uint32_t s = k % kStages, use = k / kStages;
      if (k >= kStages && !bounded_wait_warp(bars + 8 * (kStages + s), (use & 1u) ^ 1u, limit, abort_flag)) {
        live = false;
        break;
      }
      const uint32_t r0 = tile * T::TILE;
      const uint32_t nr = rows - r0 < static_cast<uint32_t>(T::TILE) ? rows - r0 : T::TILE;
      const uint32_t full = bars + 8 * s;
      if (lane == 0) {  // the copies first, so that the slot lookups below overlap them
        mbar_expect_tx(full, nr * (bcast ? T::ROW_B - 4 * T::R : T::ROW_B));
        if (!p.stall_loads) {
          const uint32_t dst = stage0 + s * T::STAGE_B;
          bulk_load(dst, p.kv + static_cast<size_t>(r0) * T::DKV, nr * T::DKV * 2, full);
          if (VARIANT == 2) bulk_load(dst + T::KV_B, p.v + static_cast<size_t>(r0) * T::DV, nr * T::DV * 2, full);
          if (!bcast) {
            bulk_load(dst + T::KV_B + T::V_B, p.cos + static_cast<size_t>(r0) * T::R, nr * T::R * 2, full);
            bulk_load(dst + T::KV_B + T::V_B + T::CS_B, p.sin + static_cast<size_t>(r0) * T::R, nr * T::R * 2, full);
          }
        }
      }
      if (lane < static_cast<int>(nr)) {  // row r0 + lane: its head and its token's index entry
        const uint32_t r = r0 + lane;
        const uint32_t bn = r / S, sq = r - bn * S;
        const uint32_t b = bn / N;
        int64_t ipos = static_cast<int64_t>(b) * S + sq;
        int32_t ax = 0;
        if (GEN && p.mode == kModeNorm) ax = static_cast<int32_t>(b);
        if (GEN && p.mode == kModePaBlkBnsd) {
          const uint32_t blk = aux.bs_shift >= 0 ? sq >> aux.bs_shift : sq / static_cast<uint32_t>(p.block_size);
          ipos = static_cast<int64_t>(b) * aux.blocks_per_batch + blk;
          ax = static_cast<int32_t>(sq - blk * static_cast<uint32_t>(p.block_size));
        }
        slot_s[s * T::TILE + lane] = __ldg(p.index + ipos);
        head_s[s * T::TILE + lane] = static_cast<int32_t>(bn - b * N);
        aux_s[s * T::TILE + lane] = ax;
        bn_s[s * T::TILE + lane] = static_cast<int32_t>(bn);
      }
      mbar_arrive(full);  // each lane releases its own writes above
    }
    if (!live && lane == 0) atomicExch(p.status, 1);
    // leave only when no copy into this block's shared memory can still be in flight
    if (lane == 0) {
      for (uint32_t u = k > static_cast<uint32_t>(kStages) ? k - kStages : 0; u < k; ++u) {
        if (!bounded_drain(bars + 8 * (u % kStages), (u / kStages) & 1u, limit)) atomicExch(p.status, 1);
      }
    }
    return;
  }

  // consumers: the quantisation tables first (the producer's first copies are already
  // in flight), then a barrier among the consumer warps only; every consumer thread
  // reaches it, since nothing before it can leave early
  if (p.kq) fill_table(ks, ko, p.k_scale, p.k_offset, heads, T::KW, kl, p.k_scalar != 0, threadIdx.x,
                       T::CWARPS * 32);
  if (p.vq) fill_table(vs, vo, p.v_scale, p.v_offset, heads, T::CW, vl, p.v_scalar != 0, threadIdx.x,
                       T::CWARPS * 32);
  asm volatile("bar.sync 1, %0;" ::"r"(T::CWARPS * 32) : "memory");
  const int g = lane / T::LPR, j = lane % T::LPR;
  uint4 gam[T::CPL];
#pragma unroll
  for (int i = 0; i < T::CPL; ++i) gam[i] = __ldg(reinterpret_cast<const uint4*>(p.gamma + 8 * (j + T::LPR * i)));
  const int64_t slots = GEN && p.mode == kModeNorm ? p.cache_seq : p.block_num * p.block_size;
  const KvRows<VARIANT, T::LPR, T::CPL, F16, GEN, true> w{
      p, aux, j, T::DKV, T::DV, T::R, T::RMS, T::RMS / 8, VARIANT == 2 ? T::CW / 8 : 0, T::R / 8, T::R / 2,
      T::KW, T::CW, slots, gam, QuantTab{ks, ko, kl.odd, kl.step, kl.stride},
      QuantTab{vs, vo, vl.odd, vl.step, vl.stride}};
  const uint4 z = make_uint4(0, 0, 0, 0);
  uint32_t k = 0;
  for (uint32_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++k) {
    const uint32_t s = k % kStages, use = k / kStages;
    if (!bounded_wait_warp(bars + 8 * s, use & 1u, limit, abort_flag)) {
      if (lane == 0) atomicExch(p.status, 1);
      return;
    }
    const uint8_t* st = smem + pl.stages + s * T::STAGE_B;
    const uint32_t r0 = tile * T::TILE;
#pragma unroll
    for (int step = 0; step < T::STEPS; ++step) {
      const int lr = (warp * T::STEPS + step) * T::RPG + g;  // row within the tile
      RowIn<T::CPL> in;
      const uint8_t* x = st + lr * T::DKV * 2;
#pragma unroll
      for (int i = 0; i < T::CPL; ++i) in.x[i] = *reinterpret_cast<const uint4*>(x + 16 * (j + T::LPR * i));
      if (VARIANT == 1) in.xr = j < T::R / 8 ? *reinterpret_cast<const uint4*>(x + 2 * T::RMS + 16 * j) : z;
      if (VARIANT == 2) {
        const uint8_t* v = st + T::KV_B + lr * T::DV * 2;
#pragma unroll
        for (int i = 0; i < T::CPL; ++i) {
          const int ch = j + T::LPR * i;
          in.v[i] = ch < T::DV / 8 ? *reinterpret_cast<const uint4*>(v + 16 * ch) : z;
        }
      }
      if (j < T::R / 8) {
        if (bcast) {  // cos/sin [B, N, 1, R]: the row of this (b, n), from the cache hierarchy
          const size_t off = static_cast<size_t>(bn_s[s * T::TILE + lr]) * T::R;
          const uint16_t* cg = p.cos + off;
          const uint16_t* sg = p.sin + off;
          in.c1 = __ldg(reinterpret_cast<const uint2*>(cg + 4 * j));
          in.c2 = __ldg(reinterpret_cast<const uint2*>(cg + T::R / 2 + 4 * j));
          in.s1 = __ldg(reinterpret_cast<const uint2*>(sg + 4 * j));
          in.s2 = __ldg(reinterpret_cast<const uint2*>(sg + T::R / 2 + 4 * j));
        } else {
          const uint8_t* cs = st + T::KV_B + T::V_B + lr * T::R * 2;
          const uint8_t* sn = cs + T::CS_B;
          in.c1 = *reinterpret_cast<const uint2*>(cs + 8 * j);
          in.c2 = *reinterpret_cast<const uint2*>(cs + T::R + 8 * j);
          in.s1 = *reinterpret_cast<const uint2*>(sn + 8 * j);
          in.s2 = *reinterpret_cast<const uint2*>(sn + T::R + 8 * j);
        }
      }
      in.slot = slot_s[s * T::TILE + lr];
      in.n = head_s[s * T::TILE + lr];
      in.aux = GEN ? aux_s[s * T::TILE + lr] : 0;
      const uint32_t row = r0 + lr;
      w.process(in, row, row < rows);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (kStages + s));
  }
}

template <int VARIANT, bool F16, bool GEN>
cudaError_t launch_staged(const KvLaunch& L, const KvAux& aux, cudaStream_t st) {
  using T = StagedShape<VARIANT>;
  auto kernel = kv_staged_kernel<VARIANT, F16, GEN>;
  const StagedPlan pl =
      staged_plan(static_cast<uint32_t>(quant_table_bytes(L, L.kq != 0, L.vq != 0, T::SPLIT)), T::STAGE_B, T::TILE);
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(pl.total));
  if (e != cudaSuccess) return e;
  const int64_t rows = L.B * L.N * L.S;
  const uint32_t tiles = static_cast<uint32_t>((rows + T::TILE - 1) / T::TILE);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, T::THREADS, pl.total) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t cap = static_cast<int64_t>(per_sm) * device_sm_count();
  const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
  kernel<<<grid, T::THREADS, pl.total, st>>>(L, aux, tiles);
  return cudaGetLastError();
}

// persistent grid: as many blocks as fit on the GPU at once, capped by the row count
template <typename K>
unsigned persistent_grid(K kernel, int64_t rows, size_t smem) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (rows + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(per_sm) * device_sm_count();
  return static_cast<unsigned>(want < cap ? want : cap);
}

template <int VARIANT, int LPR, int CPL, bool F16, bool GEN>
cudaError_t launch_one(const KvLaunch& L, const KvAux& aux, cudaStream_t st) {
  auto kernel = kv_rms_norm_rope_cache_kernel<VARIANT, LPR, CPL, F16, GEN>;
  const size_t smem = quant_table_bytes(L, L.kq != 0, L.vq != 0, true);
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = persistent_grid(kernel, L.B * L.N * L.S, smem);
  kernel<<<grid, kThreads, smem, st>>>(L, aux);
  return cudaGetLastError();
}

// lane layouts built: 8 lanes per row with 1-4 chunks each, or 16 / 32 lanes with 4
template <int VARIANT, bool F16, bool GEN>
cudaError_t launch_layout(const KvLaunch& L, const KvAux& aux, int lpr, int cpl, cudaStream_t st) {
  if (lpr == 8) {
    switch (cpl) {
      case 1: return launch_one<VARIANT, 8, 1, F16, GEN>(L, aux, st);
      case 2: return launch_one<VARIANT, 8, 2, F16, GEN>(L, aux, st);
      case 3: return launch_one<VARIANT, 8, 3, F16, GEN>(L, aux, st);
      case 4: return launch_one<VARIANT, 8, 4, F16, GEN>(L, aux, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (lpr == 16) return launch_one<VARIANT, 16, 4, F16, GEN>(L, aux, st);
  if (lpr == 32) return launch_one<VARIANT, 32, 4, F16, GEN>(L, aux, st);
  return cudaErrorInvalidValue;
}

// the pipelined kernel, when the call has one of its row shapes and the status word
// its waits report to is known
template <int VARIANT, bool F16>
bool launch_fixed(const KvLaunch& L, const KvAux& aux, int lpr, int cpl, bool gen, cudaStream_t st,
                  cudaError_t* err) {
  const bool shape = VARIANT == 1 ? L.Dkv == RowShape<1>::dkv && L.R == RowShape<1>::r && lpr == 16 && cpl == 4
                                   : L.Dkv == RowShape<2>::dkv && L.Dv == RowShape<2>::dv && L.R == RowShape<2>::r &&
                                         lpr == 8 && cpl == 3;
  if (!shape || L.status == nullptr || L.B * L.N * L.S >= (int64_t(1) << 31) - StagedShape<VARIANT>::TILE)
    return false;
  *err = gen ? launch_staged<VARIANT, F16, true>(L, aux, st) : launch_staged<VARIANT, F16, false>(L, aux, st);
  return true;
}

template <int VARIANT>
cudaError_t launch_variant(const KvLaunch& L, const KvAux& aux, int lpr, int cpl, cudaStream_t st) {
  const bool gen = (L.mode != kModePa && L.mode != kModePaBnsd) || L.rope_bcast ||
                   L.kq == kQuantE4m3 || L.kq == kQuantE5m2 || L.vq == kQuantE4m3 || L.vq == kQuantE5m2;
  cudaError_t err = cudaSuccess;
  if (L.f16 ? launch_fixed<VARIANT, true>(L, aux, lpr, cpl, gen, st, &err)
            : launch_fixed<VARIANT, false>(L, aux, lpr, cpl, gen, st, &err))
    return err;
  if (L.f16) return gen ? launch_layout<VARIANT, true, true>(L, aux, lpr, cpl, st)
                        : launch_layout<VARIANT, true, false>(L, aux, lpr, cpl, st);
  return gen ? launch_layout<VARIANT, false, true>(L, aux, lpr, cpl, st)
             : launch_layout<VARIANT, false, false>(L, aux, lpr, cpl, st);
}

}  // namespace

int32_t* kv_status_word() {
  static std::atomic<int32_t*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  if (dev < 64) {
    if (int32_t* q = cache[dev].load()) return q;
  }
  void* q = nullptr;
  if (cudaGetSymbolAddress(&q, g_kv_status) != cudaSuccess) return nullptr;
  if (dev < 64) cache[dev].store(static_cast<int32_t*>(q));
  return static_cast<int32_t*>(q);
}

cudaError_t launch_kv_rms_norm_rope_cache(const KvLaunch& L, cudaStream_t stream) {
  const int64_t rms = L.variant == 1 ? L.Dkv - L.R : L.Dkv;
  int64_t chunks = rms / 8;
  if (L.variant == 2 && L.Dv / 8 > chunks) chunks = L.Dv / 8;  // v_optional rides the same lanes
  const int64_t rope_lanes = L.R / 8;
  // the fewest lanes per row that hold the RoPE pairs and at most 4 chunks each
  // (8 lanes: as many chunks as needed; 16 or 32 lanes: 4)
  int lpr = 0, cpl = 0;
  for (int cand : {8, 16, 32}) {
    const int64_t c = (chunks + cand - 1) / cand;
    if (cand >= rope_lanes && c <= 4) {
      lpr = cand;
      cpl = cand == 8 ? static_cast<int>(c) : 4;
      break;
    }
  }
  if (lpr == 0) return cudaErrorInvalidValue;
  KvAux aux{};
  aux.inv_rms = 1.0f / static_cast<float>(rms);
  aux.bs_shift = -1;
  aux.blocks_per_batch = 0;
  if (L.mode != kModeNorm) {  // paged modes: block_size > 1 (checked by the caller)
    if ((L.block_size & (L.block_size - 1)) == 0)
      for (aux.bs_shift = 0; (int64_t(1) << aux.bs_shift) < L.block_size; ++aux.bs_shift) {
      }
    aux.blocks_per_batch = static_cast<int32_t>((L.S + L.block_size - 1) / L.block_size);
  }
  return L.variant == 1 ? launch_variant<1>(L, aux, lpr, cpl, stream)
                        : launch_variant<2>(L, aux, lpr, cpl, stream);
}

}  // namespace ra
