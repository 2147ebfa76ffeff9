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
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int kThreads = 128;
constexpr int kTok = 8;        // tokens per block
constexpr int kUnroll = 2;     // tokens whose loads are in flight together per item

__device__ __forceinline__ void lds8f(const float* p, float2 (&f)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *(reinterpret_cast<const float4*>(p) + 1);
  f[0] = make_float2(a.x, a.y); f[1] = make_float2(a.z, a.w);
  f[2] = make_float2(b.x, b.y); f[3] = make_float2(b.z, b.w);
}
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

// ---------------------------------------------------------------- pipelined kernel
// For the BSD layout with head_dim 64 or 128.  A token's Q/K columns are one
// contiguous span of `out` (20 KB for 80 heads of 128), and its partial sums,
// exponents and cos/sin rows are contiguous rows of their own, so one lane of a
// producer warp moves a token into a shared-memory stage with a handful of bulk
// copies (cp.async.bulk, completion counted by the stage's mbarrier), up to
// kSt - 1 tokens ahead.  Eight consumer warps rewrite the stage in place; when
// all eight have arrived on the stage's done barrier, one thread writes the
// span back with a bulk store and releases the stage once that store has read
// it.  Each consumer thread keeps the same 8-column offset within a head for
// every item (256 is a multiple of the items per head), so it reads its cos/sin
// once per token.  Every wait is bounded; a wait that runs out records 1 in the
// status word and the block leaves, each thread first waiting (with a limit)
// for the copies it issued.
constexpr int kSt = 3;                    // stages (measured: 3 beats 4 and 5 by 3-7 %, 2 is 40 % slower)
constexpr int kStWarps = 8;               // consumer warps
constexpr int kStThreads = (kStWarps + 1) * 32;
constexpr int kStMaxSpan = 24 * 1024;     // Q/K bytes per token the stage holds

struct StagePlan {                        // byte offsets within a stage
  uint32_t span, part, exps, cos, sin, bytes, tx;
  uint32_t span_bytes, part_bytes;
};

StagePlan stage_plan(const NormRopeLaunch& L) {
  const int h_begin = L.do_q ? 0 : L.num_q_heads;
  const int h_end = (L.num_k_heads > 0 && L.do_k) ? L.num_q_heads + L.num_k_heads : L.num_q_heads;
  StagePlan pl{};
  pl.span_bytes = static_cast<uint32_t>((h_end - h_begin) * L.head_dim * 2);
  pl.part_bytes = L.n_part_tiles > 0 ? static_cast<uint32_t>(L.part_stride) * 8u : 0u;
  pl.span = 0;
  pl.part = pl.span_bytes;
  pl.exps = pl.part + pl.part_bytes;
  pl.cos = pl.exps + static_cast<uint32_t>(L.exp_stride);
  const uint32_t cs = L.rope ? static_cast<uint32_t>(L.head_dim) * 4u : 0u;
  pl.sin = pl.cos + cs;
  pl.tx = pl.sin + cs;
  pl.bytes = (pl.tx + 127u) & ~127u;
  return pl;
}

template <int D, bool ROT>
__global__ void __launch_bounds__(kStThreads, 2)
    qk_norm_rope_staged_kernel(const NormRopeLaunch p, const StagePlan pl) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int HALF = D / 2;
  constexpr int PER_HEAD = ROT ? D / 16 : D / 8;  // 8-column items per head
  static_assert((kStWarps * 32) % PER_HEAD == 0, "a thread keeps its offset within the head");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.num_q_heads, nk = p.num_k_heads;
  const int h_begin = p.do_q ? 0 : nq;
  const int h_end = (nk > 0 && p.do_k) ? nq + nk : nq;
  const int64_t span_col = static_cast<int64_t>(h_begin) * D;
  const uint32_t bars = smem_u32(smem + kSt * pl.bytes);  // full[kSt], empty[kSt], done[kSt]
  auto full_bar = [&](uint32_t s) { return bars + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bars + 8u * (kSt + s); };
  auto done_bar = [&](uint32_t s) { return bars + 8u * (2 * kSt + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSt * pl.bytes + 3 * kSt * 8);
  const uint32_t stage0 = smem_u32(smem);
  const uint64_t limit = static_cast<uint64_t>(p.wait_ns);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(done_bar(s), kStWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kStWarps) {
    // producer: token k of this block goes to stage k % kSt
    if (lane == 0) {
      uint32_t k = 0;
      bool live = true;
      for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, ++k) {
        const uint32_t s = k % kSt, use = k / kSt;
        if (k >= kSt && !bounded_wait_one(empty_bar(s), (use & 1u) ^ 1u, limit, abort_flag)) {
          live = false;
          break;
        }
        const uint32_t full = full_bar(s), dst = stage0 + s * pl.bytes;
        mbar_arrive_expect_tx(full, pl.tx);
        if (!p.stall_loads) {
          bulk_load(dst + pl.span, p.out + t * p.I + span_col, pl.span_bytes, full);
          if (pl.part_bytes) bulk_load(dst + pl.part, p.partials + t * p.part_stride, pl.part_bytes, full);
          bulk_load(dst + pl.exps, p.exps + t * p.exp_stride, static_cast<uint32_t>(p.exp_stride), full);
          if (ROT) {
            bulk_load(dst + pl.cos, p.cos + t * D, D * 4, full);
            bulk_load(dst + pl.sin, p.sin + t * D, D * 4, full);
          }
        }
      }
      if (!live) atomicExch(p.status, 1);
      // leave only when no copy into this block's shared memory can still be in flight
      for (uint32_t u = k > static_cast<uint32_t>(kSt) ? k - kSt : 0; u < k; ++u)
        if (!bounded_drain(full_bar(u % kSt), (u / kSt) & 1u, limit)) atomicExch(p.status, 1);
    }
    return;
  }

  // consumers
  const int ct = threadIdx.x;                 // 0 .. 255
  const int u = ct % PER_HEAD;                // this thread's 8-column offset within a head
  const int items = (h_end - h_begin) * PER_HEAD;
  const int q_end = nq * D;
  const bool storer = threadIdx.x == 0;
  const float wq = static_cast<float>(nq * D), wk = static_cast<float>(nk * D);
  uint32_t k = 0;
  bool ok = true;
  for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, ++k) {
    const uint32_t s = k % kSt, use = k / kSt;
    if (!bounded_wait_warp(full_bar(s), use & 1u, limit, abort_flag)) {
      ok = false;
      break;
    }
    uint8_t* st = smem + s * pl.bytes;
    // 1b: inv_rms of the token, its partials summed lane-strided then by an xor tree
    float sq = 0.f, sk = 0.f;
    const float2* part = reinterpret_cast<const float2*>(st + pl.part);
    for (int j = lane; j < p.n_part_tiles; j += 32) {
      const float2 v = part[j];
      sq += v.x;
      sk += v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    const float inv_q = p.q_norm ? rsqrtf(sq / wq + p.eps) : 1.f;
    const float inv_k = p.k_norm ? rsqrtf(sk / wk + p.eps) : 1.f;
    const int8_t* ex = reinterpret_cast<const int8_t*>(st + pl.exps);
    float2 c_lo[4], c_hi[4], s_lo[4], s_hi[4];
    if (ROT) {
      const float* cs = reinterpret_cast<const float*>(st + pl.cos) + 8 * u;
      const float* sn = reinterpret_cast<const float*>(st + pl.sin) + 8 * u;
      lds8f(cs, c_lo);
      lds8f(cs + HALF, c_hi);
      lds8f(sn, s_lo);
      lds8f(sn + HALF, s_hi);
    }
    for (int it = ct; it < items; it += kStWarps * 32) {
      const int rel = (it / PER_HEAD) * D + 8 * u;  // column within the span
      const int col = static_cast<int>(span_col) + rel;
      const float inv = col < q_end ? inv_q : inv_k;
      uint4* lo = reinterpret_cast<uint4*>(st + pl.span + 2 * rel);
      float2 y_lo[4];
      decode8(*lo, inv * exp2_int(ex[col / kPartCols]), y_lo);
      if (ROT) {
        uint4* hi = reinterpret_cast<uint4*>(st + pl.span + 2 * (rel + HALF));
        float2 y_hi[4];
        decode8(*hi, inv * exp2_int(ex[(col + HALF) / kPartCols]), y_hi);
        float2 o_lo[4], o_hi[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          o_lo[m] = __ffma2_rn(y_lo[m], c_lo[m], __fmul2_rn(y_hi[m], make_float2(-s_lo[m].x, -s_lo[m].y)));
          o_hi[m] = __ffma2_rn(y_hi[m], c_hi[m], __fmul2_rn(y_lo[m], s_hi[m]));
        }
        *lo = pack8(o_lo);
        *hi = pack8(o_hi);
      } else {
        *lo = pack8(y_lo);
      }
    }
    // the rewritten span is read next by the bulk store (async proxy)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(done_bar(s));
    if (warp == 0) {
      int go = 1;
      if (storer) {
        go = bounded_wait_one(done_bar(s), use & 1u, limit, abort_flag) ? 1 : 0;
        if (go) {
          bulk_store(p.out + t * p.I + span_col, stage0 + s * pl.bytes + pl.span, pl.span_bytes);
          bulk_commit();
          bulk_wait_read<1>();  // the previous token's store has read its stage
          if (k > 0) mbar_arrive(empty_bar((k - 1) % kSt));
        }
      }
      go = __shfl_sync(0xffffffffu, go, 0);
      if (!go) {
        ok = false;
        break;
      }
    }
  }
  if (!ok && lane == 0) atomicExch(p.status, 1);
  if (storer) bulk_wait_all();  // this thread's stores are complete before the block ends
}

template <int D, bool ROT>
cudaError_t launch_staged(const NormRopeLaunch& L, const StagePlan& pl, cudaStream_t st) {
  auto kernel = qk_norm_rope_staged_kernel<D, ROT>;
  const size_t smem = static_cast<size_t>(kSt) * pl.bytes + 3 * kSt * 8 + 16;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kStThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t cap = static_cast<int64_t>(per_sm) * device_sm_count();
  const unsigned grid = static_cast<unsigned>(L.T < cap ? L.T : cap);
  kernel<<<grid, kStThreads, smem, st>>>(L, pl);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- pipelined kernel, NBSd
// For the NBSd layout out [I / d, T, d] with head_dim 64 or 128.  The rewritten
// heads are consecutive planes of that stack, so TB consecutive tokens of up to
// 16 consecutive heads are one 3-D box [d, TB, 16] of it: one tensor copy (TMA)
// moves a box into a stage and one tensor store writes it back, the hardware
// doing the plane strides.  The tokens' partial sums, exponents and cos/sin rows
// are contiguous rows and come in with bulk copies, as in the BSD kernel.  A
// stage holds TB tokens of every rewritten head; each consumer thread keeps one
// token and one 8-column offset within a head for the whole stage, so it reads
// its cos/sin and its token's inv_rms once per stage.  Boxes that run past the
// last token or the last rewritten head are zero-filled on load and clipped on
// store, so no other plane is touched.  Every wait is bounded, as in the BSD kernel.
constexpr int kNbHeads = 16;               // heads per tensor box, at most
constexpr int kNbSt = 3;                   // stages
constexpr int kNbWarps = 8;                // consumer warps
constexpr int kNbThreads = (kNbWarps + 1) * 32;
constexpr int kNbBlocks = 3;               // blocks per SM
// stage bytes of a block, at most: three blocks of three 1-token stages per SM
// measured 0.514 ms at 720p against 0.58-0.61 ms for one block of three 2-token
// stages, 0.61 ms for two blocks of two 2-token stages, 0.82 ms for 4-token stages
constexpr uint32_t kNbSmem = 72u * 1024;

struct NbPlan {                            // byte offsets within a stage
  uint32_t tb, hb, nbox, nh;               // tokens per stage, heads per box, boxes, rewritten heads
  uint32_t box_bytes, part, exps, cos, sin, bytes;
  uint32_t part_row, exp_row, cs_row;      // per-token bytes of each side row
};

NbPlan nb_plan(const NormRopeLaunch& L, uint32_t tb) {
  const int h_begin = L.do_q ? 0 : L.num_q_heads;
  const int h_end = (L.num_k_heads > 0 && L.do_k) ? L.num_q_heads + L.num_k_heads : L.num_q_heads;
  NbPlan pl{};
  pl.tb = tb;
  pl.nh = static_cast<uint32_t>(h_end - h_begin);
  pl.hb = pl.nh < static_cast<uint32_t>(kNbHeads) ? pl.nh : static_cast<uint32_t>(kNbHeads);
  pl.nbox = (pl.nh + pl.hb - 1) / pl.hb;
  pl.box_bytes = pl.hb * tb * static_cast<uint32_t>(L.head_dim) * 2u;
  pl.part_row = L.n_part_tiles > 0 ? static_cast<uint32_t>(L.part_stride) * 8u : 0u;
  pl.exp_row = static_cast<uint32_t>(L.exp_stride);
  pl.cs_row = L.rope ? static_cast<uint32_t>(L.head_dim) * 4u : 0u;
  auto up = [](uint32_t x) { return (x + 127u) & ~127u; };
  pl.part = pl.nbox * pl.box_bytes;
  pl.exps = up(pl.part + tb * pl.part_row);
  pl.cos = up(pl.exps + tb * pl.exp_row);
  pl.sin = up(pl.cos + tb * pl.cs_row);
  pl.bytes = up(pl.sin + tb * pl.cs_row);
  return pl;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const void* map, uint32_t src, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}

template <int D, bool ROT>
__global__ void __launch_bounds__(kNbThreads, kNbBlocks)
    qk_norm_rope_nbsd_kernel(const NormRopeLaunch p, const NbPlan pl, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int HALF = D / 2;
  constexpr int PER_HEAD = ROT ? D / 16 : D / 8;  // 8-column items per head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.num_q_heads, nk = p.num_k_heads;
  const int h_begin = p.do_q ? 0 : nq;
  const int TB = static_cast<int>(pl.tb);
  const uint32_t units = static_cast<uint32_t>((p.T + TB - 1) / TB);
  const uint32_t bars = smem_u32(smem + kNbSt * pl.bytes);  // full[kNbSt], empty[kNbSt], done[kNbSt]
  auto full_bar = [&](uint32_t s) { return bars + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bars + 8u * (kNbSt + s); };
  auto done_bar = [&](uint32_t s) { return bars + 8u * (2 * kNbSt + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kNbSt * pl.bytes + 3 * kNbSt * 8);
  const uint32_t stage0 = smem_u32(smem);
  const uint64_t limit = static_cast<uint64_t>(p.wait_ns);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNbSt; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(done_bar(s), kNbWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmap);
  }
  __syncthreads();

  if (warp == kNbWarps) {
    // producer: unit (TB tokens) k of this block goes to stage k % kNbSt
    if (lane == 0) {
      uint32_t k = 0;
      bool live = true;
      for (uint32_t unit = blockIdx.x; unit < units; unit += gridDim.x, ++k) {
        const uint32_t s = k % kNbSt, use = k / kNbSt;
        if (k >= kNbSt && !bounded_wait_one(empty_bar(s), (use & 1u) ^ 1u, limit, abort_flag)) {
          live = false;
          break;
        }
        const int64_t t0 = static_cast<int64_t>(unit) * TB;
        const uint32_t nt = static_cast<uint32_t>(p.T - t0 < TB ? p.T - t0 : TB);
        const uint32_t full = full_bar(s), dst = stage0 + s * pl.bytes;
        // a box counts its full size, zero-filled past the last token or head
        mbar_arrive_expect_tx(full, pl.nbox * pl.box_bytes + nt * (pl.part_row + pl.exp_row + 2 * pl.cs_row));
        if (!p.stall_loads) {
          for (uint32_t b = 0; b < pl.nbox; ++b)
            tma_load_3d(dst + b * pl.box_bytes, &tmap, full, 0, static_cast<int32_t>(t0),
                        static_cast<int32_t>(b * pl.hb));
          if (pl.part_row) bulk_load(dst + pl.part, p.partials + t0 * p.part_stride, nt * pl.part_row, full);
          bulk_load(dst + pl.exps, p.exps + t0 * p.exp_stride, nt * pl.exp_row, full);
          if (ROT) {
            bulk_load(dst + pl.cos, p.cos + t0 * D, nt * pl.cs_row, full);
            bulk_load(dst + pl.sin, p.sin + t0 * D, nt * pl.cs_row, full);
          }
        }
      }
      if (!live) atomicExch(p.status, 1);
      // leave only when no copy into this block's shared memory can still be in flight
      for (uint32_t u = k > static_cast<uint32_t>(kNbSt) ? k - kNbSt : 0; u < k; ++u)
        if (!bounded_drain(full_bar(u % kNbSt), (u / kNbSt) & 1u, limit)) atomicExch(p.status, 1);
    }
    return;
  }

  // consumers
  const int ct = threadIdx.x;                                // 0 .. 32 * kNbWarps - 1
  const int u = ct % PER_HEAD;                               // this thread's 8-column offset within a head
  const int tok = (ct / PER_HEAD) % TB;                      // and its token within the stage
  const int hstep = (kNbWarps * 32) / (PER_HEAD * TB);       // heads between this thread's items
  const int head0 = ct / (PER_HEAD * TB);
  const int q_end = nq * D;
  const bool storer = threadIdx.x == 0;
  const float wq = static_cast<float>(nq * D), wk = static_cast<float>(nk * D);
  uint32_t k = 0;
  bool ok = true;
  for (uint32_t unit = blockIdx.x; unit < units; unit += gridDim.x, ++k) {
    const uint32_t s = k % kNbSt, use = k / kNbSt;
    if (!bounded_wait_warp(full_bar(s), use & 1u, limit, abort_flag)) {
      ok = false;
      break;
    }
    uint8_t* st = smem + s * pl.bytes;
    const int64_t t0 = static_cast<int64_t>(unit) * TB;
    const int nt = static_cast<int>(p.T - t0 < TB ? p.T - t0 : TB);
    // 1b: inv_rms of this thread's token; every warp sums the stage's partials in the
    // same fixed order (lane-strided, then an xor tree)
    float inv_q = 1.f, inv_k = 1.f;
    const float2* part = reinterpret_cast<const float2*>(st + pl.part);
    for (int tt = 0; tt < nt; ++tt) {
      float sq = 0.f, sk = 0.f;
      for (int j = lane; j < p.n_part_tiles; j += 32) {
        const float2 v = part[tt * p.part_stride + j];
        sq += v.x;
        sk += v.y;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      if (tt == tok) {
        inv_q = p.q_norm ? rsqrtf(sq / wq + p.eps) : 1.f;
        inv_k = p.k_norm ? rsqrtf(sk / wk + p.eps) : 1.f;
      }
    }
    if (tok < nt) {
      const int8_t* ex = reinterpret_cast<const int8_t*>(st + pl.exps) + tok * pl.exp_row;
      float2 c_lo[4], c_hi[4], s_lo[4], s_hi[4];
      if (ROT) {
        const float* cs = reinterpret_cast<const float*>(st + pl.cos + tok * pl.cs_row) + 8 * u;
        const float* sn = reinterpret_cast<const float*>(st + pl.sin + tok * pl.cs_row) + 8 * u;
        lds8f(cs, c_lo);
        lds8f(cs + HALF, c_hi);
        lds8f(sn, s_lo);
        lds8f(sn + HALF, s_hi);
      }
      for (int head = head0; head < static_cast<int>(pl.nh); head += hstep) {
        const int col = (h_begin + head) * D + 8 * u;
        const float inv = col < q_end ? inv_q : inv_k;
        uint4* lo = reinterpret_cast<uint4*>(st + 2 * ((head * TB + tok) * D + 8 * u));
        float2 y_lo[4];
        decode8(*lo, inv * exp2_int(ex[col / kPartCols]), y_lo);
        if (ROT) {
          uint4* hi = lo + HALF / 8;
          float2 y_hi[4];
          decode8(*hi, inv * exp2_int(ex[(col + HALF) / kPartCols]), y_hi);
          float2 o_lo[4], o_hi[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            o_lo[m] = __ffma2_rn(y_lo[m], c_lo[m], __fmul2_rn(y_hi[m], make_float2(-s_lo[m].x, -s_lo[m].y)));
            o_hi[m] = __ffma2_rn(y_hi[m], c_hi[m], __fmul2_rn(y_lo[m], s_hi[m]));
          }
          *lo = pack8(o_lo);
          *hi = pack8(o_hi);
        } else {
          *lo = pack8(y_lo);
        }
      }
    }
    // the rewritten boxes are read next by the tensor stores (async proxy)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(done_bar(s));
    if (warp == 0) {
      int go = 1;
      if (storer) {
        go = bounded_wait_one(done_bar(s), use & 1u, limit, abort_flag) ? 1 : 0;
        if (go) {
          for (uint32_t b = 0; b < pl.nbox; ++b)
            tma_store_3d(&tmap, stage0 + s * pl.bytes + b * pl.box_bytes, 0, static_cast<int32_t>(t0),
                         static_cast<int32_t>(b * pl.hb));
          bulk_commit();
          bulk_wait_read<1>();  // the previous unit's stores have read their stage
          if (k > 0) mbar_arrive(empty_bar((k - 1) % kNbSt));
        }
      }
      go = __shfl_sync(0xffffffffu, go, 0);
      if (!go) {
        ok = false;
        break;
      }
    }
  }
  if (!ok && lane == 0) atomicExch(p.status, 1);
  if (storer) bulk_wait_all();  // this thread's stores are complete before the block ends
}

size_t nb_smem(const NbPlan& pl) { return static_cast<size_t>(kNbSt) * pl.bytes + 3 * kNbSt * 8 + 16; }

// the largest stage of 8, 4, 2 or 1 tokens whose ring fits the budget (0: none fits)
uint32_t nb_tokens(const NormRopeLaunch& L) {
  for (uint32_t tb = 8; tb >= 1; tb /= 2)
    if (tb <= L.T && nb_smem(nb_plan(L, tb)) <= kNbSmem) return tb;
  return 0;
}

template <int D, bool ROT>
cudaError_t launch_nbsd(const NormRopeLaunch& L, const NbPlan& pl, cudaStream_t st) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorInvalidValue;
  const int h_begin = L.do_q ? 0 : L.num_q_heads;
  // the rewritten heads' planes as a [nh, T, D] stack of 16-bit values
  CUtensorMap tmap;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L.T), pl.nh};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(L.T) * D * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(D), pl.tb, pl.hb};
  cuuint32_t estr[3] = {1, 1, 1};
  void* base = L.out + static_cast<size_t>(h_begin) * L.T * D;
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  auto kernel = qk_norm_rope_nbsd_kernel<D, ROT>;
  const size_t smem = nb_smem(pl);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kNbThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t units = (L.T + pl.tb - 1) / pl.tb;
  const int64_t cap = static_cast<int64_t>(per_sm) * device_sm_count();
  kernel<<<static_cast<unsigned>(units < cap ? units : cap), kNbThreads, smem, st>>>(L, pl, tmap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope(const NormRopeLaunch& L, cudaStream_t stream) {
  const StagePlan pl = stage_plan(L);
  const bool staged = !L.nbsd && L.status != nullptr && (L.head_dim == 64 || L.head_dim == 128) &&
                      pl.span_bytes > 0 && pl.span_bytes <= static_cast<uint32_t>(kStMaxSpan) &&
                      L.exp_stride > 0 && L.exp_stride % 16 == 0 && L.part_stride % 2 == 0 &&
                      L.I % 8 == 0 && L.T < (int64_t(1) << 31);
  if (staged) {
    if (L.head_dim == 128) return L.rope ? launch_staged<128, true>(L, pl, stream) : launch_staged<128, false>(L, pl, stream);
    return L.rope ? launch_staged<64, true>(L, pl, stream) : launch_staged<64, false>(L, pl, stream);
  }
  if (L.nbsd && L.status != nullptr && (L.head_dim == 64 || L.head_dim == 128) && pl.span_bytes > 0 &&
      L.exp_stride > 0 && L.exp_stride % 16 == 0 && L.part_stride % 2 == 0 && L.T < (int64_t(1) << 31)) {
    const uint32_t tb = nb_tokens(L);
    if (tb > 0) {
      const NbPlan np = nb_plan(L, tb);
      if (L.head_dim == 128) return L.rope ? launch_nbsd<128, true>(L, np, stream) : launch_nbsd<128, false>(L, np, stream);
      return L.rope ? launch_nbsd<64, true>(L, np, stream) : launch_nbsd<64, false>(L, np, stream);
    }
  }
  const int64_t blocks = (L.T + kTok - 1) / kTok;
  qk_norm_rope_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(L);
  return cudaGetLastError();
}

}  // namespace ra
