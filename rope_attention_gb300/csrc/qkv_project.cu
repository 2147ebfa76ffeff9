// K1: block-scaled FP8 projection with the dequant / bias / sum-of-squares epilogue.
//
// Computes, for the fused QKV projection of the AWS Neuron page "Kernel
// reference: qkv_cte" (section "Upstream behavior": O[S, I] = A[S, H] @ W[H, I]
// (+ bias); Pattern: the accumulator is dequantised and bias-added while it is
// read out, then stored to HBM; Design 1a: per-token sum(x^2) over the whole Q
// and K segments of the un-normalised output):
//
//   acc[t, i]     = sum_h e4m3(a[t, h]) * e4m3(w[h, i]) * 2^(e[h/32, i] - 127)
//   v[t, i]       = acc[t, i] * a_scale[t] * wch[i] + bias[i]
//   out[t, i]     = bf16(v)  for V (and any segment the second pass leaves alone),
//   out[t, i]     = fp16(z * 2^-e[t, b]) for the Q/K columns the norm/RoPE pass
//                   rewrites, z = v * gamma[i] (the segment-wide gamma of Design 1c,
//                   which commutes with the per-token inv_rms and the rotation), with
//                   one power-of-two exponent per (row, 128-column block b) chosen so
//                   the block's largest |z| lands in [2^14, 2^15): 11 significant
//                   bits in the 2 bytes the final bf16 needs
//   partial[t, j] = ( sum of v^2 over the Q columns of 128-column block j,
//                     sum of v^2 over its K columns )
//
// GB300 design (not the page's NKI schedule):
//  * CTA pairs (clusters of 2) run tcgen05.mma.cta_group::2 kind::mxf8f6f4 on
//    256 x 256 output tiles (M=256, N=256, K=32 per instruction): each CTA holds
//    128 rows of A and 128 rows (columns of the output) of W in shared memory, so
//    each SM stages 33 KB per 128-deep K step instead of the 46 KB a single-SM
//    128 x 240 tile needs; the pair's accumulator is split by rows across the
//    two SMs' TMEM;
//  * persistent pairs (one pair per two SMs), grouped rasterisation;
//  * warp 0 (both CTAs): TMA producer into a 6-stage ring; the loads of both
//    CTAs complete on the leader CTA's full barrier;
//  * warp 1: allocates TMEM (512 columns, pair-wide); in the leader CTA one
//    thread issues the MMAs and copies W's ue8m0 block scales into TMEM each
//    stage (tcgen05.cp); A's MX scale is the constant 2^0 (its fp32 row scale is
//    applied in the epilogue, since it is constant along K); commits multicast
//    to both CTAs.  With an even number of K steps it issues two stages per asm
//    block and learns whether the next two have landed from a probe issued at the
//    block's start and read at its end, so the thread never stalls on a barrier
//    read while the tensor pipe has work queued;
//  * warps 2-9 (both CTAs): epilogue, two warps per TMEM lane quadrant, each
//    owning 128 of the 256 columns; they pull the whole accumulator into
//    registers first and release TMEM before the math and stores, so the next
//    tile's MMAs start after a short drain.
// Every pipeline wait is bounded in time; on expiry a CTA records an error in
// the status word, waits (bounded) for the copies and MMAs it started, frees
// TMEM with its peer and exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int BM = 128;               // output rows per CTA (a pair covers 256)
constexpr int PAIR_M = 2 * BM;
constexpr int BN = kProjBN;           // output columns per pair tile
constexpr int BN_HALF = BN / 2;       // W rows staged per CTA
constexpr int BK = kProjBK;
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN_HALF * BK;
constexpr int SF_BYTES = kSfStageBytes;  // one stage's W scale image (see pack_sf_kernel)
constexpr uint32_t STAGE_TX = 2u * (A_BYTES + B_BYTES + SF_BYTES);  // both CTAs, on the leader's barrier
constexpr int ACC_COL = 0;
constexpr int SFA_COL = BN;           // 4 columns of A scales
constexpr int SFB_COL = BN + 8;       // two 8-column slots of W scales
constexpr int TMEM_COLS = 512;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;  // 10 warps: at most 3 per SM sub-partition, so <= 168 registers each
constexpr int EPI_COLS = BN / 2;      // columns per epilogue warp
constexpr int GROUP_M = 16;          // M-tiles per raster group: W is read from HBM once per group

constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * A_BYTES;
constexpr int SMEM_SF = SMEM_B + STAGES * B_BYTES;
constexpr int SMEM_SFA = SMEM_SF + STAGES * SF_BYTES;
constexpr int SMEM_BAR = SMEM_SFA + 512;
constexpr int NUM_BARS = 2 * STAGES + 3;
constexpr int SMEM_MISC = SMEM_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = SMEM_MISC + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack to align the base to 1024 bytes

static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms must stay aligned");
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
static_assert(SFB_COL + 16 <= TMEM_COLS, "TMEM budget");
static_assert(BN == 256 && SF_BYTES == 4096, "pair tile shape");
static_assert(kPartCols == EPI_COLS, "one partial per epilogue warp and row");

// Instruction descriptor, block-scaled kinds: A/B format E4M3 (0) in bits
// [7,10)/[10,13), K-major operands, N>>3 in [17,23), scale type UE8M0 (1) at
// bit 23, M>>4 in [24,29); the scale-factor ids go in [29,31) (A) and [4,6) (B).
constexpr uint32_t kIdesc = (uint32_t(BN >> 3) << 17) | (1u << 23) | (uint32_t(PAIR_M >> 4) << 24);

struct Params {
  CUtensorMap tmap_a;   // [T, H] bytes, box 128 x 128, 128-byte swizzle
  CUtensorMap tmap_b;   // [I, H] bytes, box 128 x 128, 128-byte swizzle
  CUtensorMap tmap_sf;  // scale images viewed as [rows, 256] bytes, box 256 x 16 (one image)
  const float* a_scale;
  const float* wch;
  const uint16_t* bias;
  uint16_t* out;
  int8_t* exps;
  float2* partials;
  int32_t* status;
  int32_t T, I, num_k, num_m, num_n;
  int32_t q_end, k_end, n_part, n_exp, part_stride, exp_stride;
  int32_t s_begin, s_end;
  const float* q_gamma;
  const float* k_gamma;
  uint64_t wait_ns;
  int32_t stall_loads;
  int32_t head_dim, nbsd;
  int32_t out32;  // out is 32-byte aligned, so every 16-column chunk is (I and head_dim are multiples of 16)
  int32_t ph_begin, ph_end, ph_carry;
  const float* ph_q_gamma;
  const float* ph_k_gamma;
  float eps;
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& m_blk, int& n_tile) {
  const int per_group = GROUP_M * num_n;
  const int group = tile / per_group;
  const int first_m = group * GROUP_M;
  const int gm = min(GROUP_M, num_m - first_m);
  const int local = tile - group * per_group;
  m_blk = first_m + local % gm;
  n_tile = local / gm;
}

// single-thread bounded wait; false when this or another role gave up
__device__ bool wait_one(uint32_t bar, uint32_t parity, uint64_t limit, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// single-thread bounded wait on a stage pair's two full barriers (same parity); each
// poll probes both in one shared-memory round trip, not one after the other
__device__ bool wait_pair(uint32_t bar0, uint32_t parity, uint64_t limit, volatile int* abort_flag) {
  if (mbar_test_wait_pair(bar0, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_wait_pair(bar0, parity)) return true;
    if ((i & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// warp-collective bounded wait: every lane returns the same answer
__device__ bool wait_warp(uint32_t bar, uint32_t parity, uint64_t limit, volatile int* abort_flag) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((i & 31u) == 31u) {
      int give_up = 0;
      if (lane_id() == 0) {
        const uint64_t t = globaltimer_ns();
        if (t0 == 0) t0 = t;
        else if (*abort_flag || t - t0 > limit) give_up = 1;
      }
      give_up = __shfl_sync(0xffffffffu, give_up, 0);
      if (give_up) {
        if (lane_id() == 0) *abort_flag = 1;
        return false;
      }
    }
  }
}

// bounded wait used only while tearing down (ignores the abort flag)
__device__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit) return;
  }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// One (lo, hi) pair of 16-column chunks of a head for the per-head norm (qkv_cte
// page, Design 1: the upstream qk-norm, each head's slice by its own RMS, with a
// [head_dim] gamma) when the call has no RoPE: r holds v (after dequant and bias);
// the pair is normed and stored as bf16.  (With RoPE a per-head segment is normed
// in the pass-1 loop below and carried to the RoPE pass instead.)
template <int D>
__device__ __forceinline__ void per_head_pair(uint32_t (&r)[EPI_COLS], int lo_c, int hi_c, int jc, float inv,
                                              const float* g, uint16_t* dst_lo, uint16_t* dst_hi) {
  const float2 inv2 = make_float2(inv, inv);
  // two halves of 8 columns each, so that few values are live beside the accumulator
#pragma unroll
  for (int half8 = 0; half8 < 2; ++half8) {
    asm volatile("" ::: "memory");  // keep this half's side loads from being hoisted
    const int j = jc + 8 * half8;
    float2 y_lo[4], y_hi[4];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float4 gl = __ldg(reinterpret_cast<const float4*>(g + j) + q);
      const float4 gh = __ldg(reinterpret_cast<const float4*>(g + j + D / 2) + q);
      const int k = 8 * half8 + 4 * q;
      y_lo[2 * q] = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(r[lo_c * 16 + k]), __uint_as_float(r[lo_c * 16 + k + 1])), inv2), make_float2(gl.x, gl.y));
      y_lo[2 * q + 1] = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(r[lo_c * 16 + k + 2]), __uint_as_float(r[lo_c * 16 + k + 3])), inv2), make_float2(gl.z, gl.w));
      y_hi[2 * q] = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(r[hi_c * 16 + k]), __uint_as_float(r[hi_c * 16 + k + 1])), inv2), make_float2(gh.x, gh.y));
      y_hi[2 * q + 1] = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(r[hi_c * 16 + k + 2]), __uint_as_float(r[hi_c * 16 + k + 3])), inv2), make_float2(gh.z, gh.w));
    }
    reinterpret_cast<uint4*>(dst_lo)[half8] =
        make_uint4(pack_bf16x2(y_lo[0].x, y_lo[0].y), pack_bf16x2(y_lo[1].x, y_lo[1].y),
                   pack_bf16x2(y_lo[2].x, y_lo[2].y), pack_bf16x2(y_lo[3].x, y_lo[3].y));
    reinterpret_cast<uint4*>(dst_hi)[half8] =
        make_uint4(pack_bf16x2(y_hi[0].x, y_hi[0].y), pack_bf16x2(y_hi[1].x, y_hi[1].y),
                   pack_bf16x2(y_hi[2].x, y_hi[2].y), pack_bf16x2(y_hi[3].x, y_hi[3].y));
  }
}

// PHD: head_dim of the per-head norm path built into the epilogue, 0 for none (a
// separate instantiation, so the across-heads kernel keeps its register allocation)
template <int PHD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    qkv_project_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sA = s_base + SMEM_A;
  const uint32_t sB = s_base + SMEM_B;
  const uint32_t sSF = s_base + SMEM_SF;
  const uint32_t sSFA = s_base + SMEM_SFA;
  const uint32_t bar0 = s_base + SMEM_BAR;
  const uint32_t accf_bar = bar0 + 8u * (2 * STAGES);
  const uint32_t acce_bar = bar0 + 8u * (2 * STAGES + 1);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_MISC + 4);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = leader of the pair
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);
  // The leader stages W rows [0, 128) of the tile and the peer rows [128, 256); both
  // stage the full 256-column scale image, since each SM's MMA half applies the
  // scales of all N columns.
  const uint32_t b_half = rank;
  const uint64_t drain_ns = 200000000ull;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, 2 * NUM_EPI_WARPS);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&p.tmap_a);
    prefetch_tensormap(&p.tmap_b);
    prefetch_tensormap(&p.tmap_sf);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (threadIdx.x >= 64 && threadIdx.x < 64 + 128) {
    // A's MX scale factors: ue8m0 127 (= 1.0) for every row and block
    reinterpret_cast<uint32_t*>(smem + SMEM_SFA)[threadIdx.x - 64] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int num_tiles = p.num_m * p.num_n;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0 && !p.stall_loads) {
      const uint32_t leader_full0 = map_to_rank(full_bar(0), 0);
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        int mb, nt;
        tile_coords(tile, p.num_m, p.num_n, mb, nt);
        for (int kb = 0; kb < p.num_k; ++kb) {
          if (!wait_one(empty_bar(stage), phase ^ 1u, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(full_bar(stage), STAGE_TX);
          const uint32_t fb = leader_full0 + 8u * stage;
          tma_load_2d_pair(sA + stage * A_BYTES, &p.tmap_a, fb, kb * BK, mb * PAIR_M + rank * BM);
          tma_load_2d_pair(sB + stage * B_BYTES, &p.tmap_b, fb, kb * BK, nt * BN + b_half * BN_HALF);
          const int sf_row = (nt * p.num_k + kb) * (SF_BYTES / 256);
          const uint32_t sf_dst = sSF + stage * SF_BYTES;
          tma_load_2d_pair(sf_dst, &p.tmap_sf, fb, 0, sf_row);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // the leader's full barriers count both CTAs' bytes: let every armed load land
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) wait_drain(full_bar(s), (armed_parity >> s) & 1u, drain_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (leader && lane == 0) {
      tc_cp_pair_32x128b_warpx4(tmem + SFA_COL, sdesc_scale_rows(sSFA));
      // shared-memory descriptors of stage 0; a stage or a 32-byte K step only moves
      // the start-address field (bits [0,14), in 16-byte units, no carry out of it
      // since every address here is below 2^18), so the loop steps them by addition
      const uint64_t a_desc0 = sdesc_kmajor_sw128(sA);
      const uint64_t b_desc0 = sdesc_kmajor_sw128(sB);
      const uint64_t sf_desc0 = sdesc_scale_image(sSF);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      // An even number of K steps per tile keeps every tile (and so every pair of
      // stages) starting on an even stage of the even-length ring: those calls issue
      // two stages per asm block with a look-ahead probe of the next pair's barriers
      // (tc_mma_stage_pair_mxf8); other calls one stage per block with a probe of the
      // next stage (tc_mma_stage_mxf8).  `ready` is the probe's answer for what is
      // about to be issued; when it is false the issuer takes a bounded wait first.
      const bool paired = (p.num_k & 1) == 0;
      static_assert(STAGES % 2 == 0, "stage pairs must not wrap the ring");
      static_assert(A_BYTES == 16384 && B_BYTES == 16384 && SF_BYTES == 4096 && BK == 128,
                    "tc_mma_stage_pair_mxf8 steps stages by 16 KB operands, 4 KB scale images, 4 K steps");
      bool ready = false;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs, ++local) {
        if (!wait_one(acce_bar, (static_cast<uint32_t>(local) & 1u) ^ 1u, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; paired && kb < p.num_k; kb += 2) {
          if (!ready && !wait_pair(full_bar(stage), phase, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nstage = stage + 2 == STAGES ? 0 : stage + 2;
          const uint32_t nphase = nstage == 0 ? phase ^ 1u : phase;
          ready = tc_mma_stage_pair_mxf8(full_bar(nstage), nphase, tmem + SFB_COL,
                                         sf_desc0 + static_cast<uint64_t>(stage * (SF_BYTES >> 4)), tmem + ACC_COL,
                                         a_desc0 + static_cast<uint64_t>(stage * (A_BYTES >> 4)),
                                         b_desc0 + static_cast<uint64_t>(stage * (B_BYTES >> 4)), kIdesc,
                                         tmem + SFA_COL, kb != 0 ? 1u : 0u, empty_bar(stage));
          stage = nstage;
          phase = nphase;
        }
        // odd number of K steps: one stage per asm block, with the same look-ahead probe
        // of the next stage; the scale slot follows the ring position, so consecutive
        // stages use different slots across tile boundaries too
        for (int kb = 0; !paired && kb < p.num_k; ++kb) {
          if (!ready && !wait_one(full_bar(stage), phase, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nstage = stage + 1 == STAGES ? 0 : stage + 1;
          const uint32_t nphase = nstage == 0 ? phase ^ 1u : phase;
          ready = tc_mma_stage_mxf8(full_bar(nstage), nphase, tmem + SFB_COL + (stage & 1) * 8,
                                    sf_desc0 + static_cast<uint64_t>(stage * (SF_BYTES >> 4)), tmem + ACC_COL,
                                    a_desc0 + static_cast<uint64_t>(stage * (A_BYTES >> 4)),
                                    b_desc0 + static_cast<uint64_t>(stage * (B_BYTES >> 4)), kIdesc, tmem + SFA_COL,
                                    kb != 0 ? 1u : 0u, empty_bar(stage));
          stage = nstage;
          phase = nphase;
        }
        if (ok) tc_commit_pair_multicast(accf_bar, 0x3);
      }
      // every MMA and copy issued here must finish before TMEM is released
      tc_commit_pair(drain_bar);
      wait_drain(drain_bar, 0, drain_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    const int quad = warp & 3;           // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int chalf = ew >> 2;           // which 128 of the tile's 256 columns
    const int row_in_cta = quad * 32 + lane;
    const uint32_t acce_leader = map_to_rank(acce_bar, 0);
    int local = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs, ++local) {
      int mb, nt;
      tile_coords(tile, p.num_m, p.num_n, mb, nt);
      if (!wait_warp(accf_bar, static_cast<uint32_t>(local) & 1u, p.wait_ns, abort_flag)) break;
      tc_fence_after();
      uint32_t r[EPI_COLS];
      const uint32_t t_base =
          tmem + ACC_COL + chalf * EPI_COLS + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll
      for (int c = 0; c < EPI_COLS / 16; ++c) tmem_ld16(t_base + c * 16, r + c * 16);
      tmem_ld_wait();
      // the accumulator is in registers: hand TMEM back to the MMA issuer now.  The
      // TMEM reads have completed (tcgen05.wait::ld), which is all the issuer needs
      // before it overwrites the accumulator, so the arrive is relaxed: a release
      // would first wait for this warp's stores of the previous tile to become
      // visible to the cluster and hold the tensor pipe idle meanwhile (3-5 %).
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader);

      const int row = mb * PAIR_M + static_cast<int>(rank) * BM + row_in_cta;
      const bool row_ok = row < p.T;
      const float as = row_ok ? __ldg(p.a_scale + row) : 0.f;
      float ssq = 0.f, ssk = 0.f;
      const size_t orow = static_cast<size_t>(row_ok ? row : 0);
      uint16_t* out_row = p.out + orow * p.I;
      const int col_base = nt * BN + chalf * EPI_COLS;
      float ph_ss[PHD > 0 ? EPI_COLS / PHD : 1];  // per-head sums of v^2 (per-head norm)
#pragma unroll
      for (int h = 0; h < (PHD > 0 ? EPI_COLS / PHD : 1); ++h) ph_ss[h] = 0.f;
      // pass 1: dequant, channel scale and bias in place (packed fp32x2 arithmetic);
      // sums of squares of v, before gamma
      const float2 as2 = make_float2(as, as);
#pragma unroll
      for (int c = 0; c < EPI_COLS / 16; ++c) {
        const int col0 = col_base + c * 16;
        if (col0 >= p.I) break;  // ragged last column tile; warp-uniform
        float2 bia[8];
        if (p.bias != nullptr) {
          const uint4* b4 = reinterpret_cast<const uint4*>(p.bias + col0);
          const uint4 t0 = __ldg(b4), t1 = __ldg(b4 + 1);
          bia[0] = bf16x2_to_float2(t0.x); bia[1] = bf16x2_to_float2(t0.y);
          bia[2] = bf16x2_to_float2(t0.z); bia[3] = bf16x2_to_float2(t0.w);
          bia[4] = bf16x2_to_float2(t1.x); bia[5] = bf16x2_to_float2(t1.y);
          bia[6] = bf16x2_to_float2(t1.z); bia[7] = bf16x2_to_float2(t1.w);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) bia[k] = make_float2(0.f, 0.f);
        }
        float2 sq2 = make_float2(0.f, 0.f);
        if (p.wch != nullptr) {
          const float4* w4 = reinterpret_cast<const float4*>(p.wch + col0);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 w = __ldg(w4 + k4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int k = 2 * k4 + h;
              const float2 acc = make_float2(__uint_as_float(r[c * 16 + 2 * k]), __uint_as_float(r[c * 16 + 2 * k + 1]));
              const float2 v = __ffma2_rn(__fmul2_rn(acc, as2), h ? make_float2(w.z, w.w) : make_float2(w.x, w.y), bia[k]);
              r[c * 16 + 2 * k] = __float_as_uint(v.x);
              r[c * 16 + 2 * k + 1] = __float_as_uint(v.y);
              sq2 = __ffma2_rn(v, v, sq2);
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 acc = make_float2(__uint_as_float(r[c * 16 + 2 * k]), __uint_as_float(r[c * 16 + 2 * k + 1]));
            const float2 v = __ffma2_rn(acc, as2, bia[k]);
            r[c * 16 + 2 * k] = __float_as_uint(v.x);
            r[c * 16 + 2 * k + 1] = __float_as_uint(v.y);
            sq2 = __ffma2_rn(v, v, sq2);
          }
        }
        if constexpr (PHD > 0) ph_ss[c / (PHD / 16)] += sq2.x + sq2.y;
        if (col0 < p.q_end) ssq += sq2.x + sq2.y;
        else if (col0 < p.k_end) ssk += sq2.x + sq2.y;
      }
      // segments with the per-head norm are finished here
      // the segment-wide gamma of the normed segments, on the columns the second
      // pass rewrites (inv_rms is one scalar per token and segment, and RoPE is
      // linear, so scaling by gamma here is exact: rot(v * inv * gamma) = inv * rot(v * gamma)),
      // and the largest |z| of the rewritten columns
      float amax = 0.f;
#pragma unroll
      for (int c = 0; c < EPI_COLS / 16; ++c) {
        const int col0 = col_base + c * 16;
        if (col0 >= p.I) break;
        if (col0 < p.s_begin || col0 >= p.s_end) continue;
        if constexpr (PHD > 0) {
          // a per-head segment carried to the RoPE pass: its norm (inv_rms of the head,
          // then the per-head gamma) is applied here, before the encoding
          if (p.ph_carry && col0 >= p.ph_begin && col0 < p.ph_end) {
            const float inv = rsqrtf(ph_ss[c / (PHD / 16)] * (1.f / PHD) + p.eps);
            const float2 inv2 = make_float2(inv, inv);
            const float4* g4 = reinterpret_cast<const float4*>((col0 < p.q_end ? p.ph_q_gamma : p.ph_k_gamma) + col0 % PHD);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const float4 t = __ldg(g4 + k4);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int k = 2 * k4 + h;
                const float2 v = make_float2(__uint_as_float(r[c * 16 + 2 * k]), __uint_as_float(r[c * 16 + 2 * k + 1]));
                const float2 z = __fmul2_rn(__fmul2_rn(v, inv2), h ? make_float2(t.z, t.w) : make_float2(t.x, t.y));
                r[c * 16 + 2 * k] = __float_as_uint(z.x);
                r[c * 16 + 2 * k + 1] = __float_as_uint(z.y);
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(__uint_as_float(r[c * 16 + j])));
            continue;
          }
        }
        const float* g = col0 < p.q_end ? p.q_gamma : p.k_gamma;
        if (g != nullptr) {
          const float4* g4 = reinterpret_cast<const float4*>(g + (col0 < p.q_end ? col0 : col0 - p.q_end));
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 t = __ldg(g4 + k4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int k = 2 * k4 + h;
              const float2 v = make_float2(__uint_as_float(r[c * 16 + 2 * k]), __uint_as_float(r[c * 16 + 2 * k + 1]));
              const float2 z = __fmul2_rn(v, h ? make_float2(t.z, t.w) : make_float2(t.x, t.y));
              r[c * 16 + 2 * k] = __float_as_uint(z.x);
              r[c * 16 + 2 * k + 1] = __float_as_uint(z.y);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(__uint_as_float(r[c * 16 + j])));
      }
      // power-of-two scale for the fp16 encoding: |z| * 2^-e < 2^15
      const int e = scale_exponent(amax);
      const float2 down2 = make_float2(exp2_int(-e), exp2_int(-e));
      // pass 2: stores (fp16 of z * 2^-e for the rewritten Q/K columns, bf16 otherwise)
#pragma unroll
      for (int c = 0; c < EPI_COLS / 16; ++c) {
        const int col0 = col_base + c * 16;
        if (col0 >= p.I) break;
        if (!row_ok) continue;
        // BSD: [T, I]; NBSd: [I / head_dim, T, head_dim] (a 16-column chunk never crosses a head)
        auto out_at = [&](int col) {
          return p.nbsd ? p.out + (static_cast<size_t>(col / p.head_dim) * p.T + orow) * p.head_dim + col % p.head_dim
                        : out_row + col;
        };
        if constexpr (PHD > 0) {
          // per-head segments: each (lo, hi) chunk pair of a head is normed, rotated and
          // stored when its lo chunk comes up
          const int hh = c / (PHD / 16), cin = c % (PHD / 16);
          const int h0 = col_base + hh * PHD;
          if (!p.ph_carry && h0 >= p.ph_begin && h0 < p.ph_end) {
            if (cin < PHD / 32) {
              const float inv = rsqrtf(ph_ss[hh] * (1.f / PHD) + p.eps);
              const float* g = h0 < p.q_end ? p.ph_q_gamma : p.ph_k_gamma;
              per_head_pair<PHD>(r, c, c + PHD / 32, cin * 16, inv, g, out_at(col0), out_at(col0 + PHD / 2));
            }
            continue;
          }
        }
        uint32_t o[8];
        if (col0 >= p.s_begin && col0 < p.s_end) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 z = __fmul2_rn(make_float2(__uint_as_float(r[c * 16 + 2 * k]), __uint_as_float(r[c * 16 + 2 * k + 1])), down2);
            o[k] = pack_f16x2(z.x, z.y);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            o[k] = pack_bf16x2(__uint_as_float(r[c * 16 + 2 * k]), __uint_as_float(r[c * 16 + 2 * k + 1]));
        }
        uint16_t* dst = out_at(col0);
        if (p.out32) {  // one 32-byte store (sm_100+): half the store instructions and transactions
          asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(o[0]), "r"(o[1]),
                       "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                       : "memory");
        } else {
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      const int blk = nt * 2 + chalf;
      if (blk < p.n_exp && row_ok)
        p.exps[static_cast<size_t>(row) * p.exp_stride + blk] = static_cast<int8_t>(e);
      const int part = nt * 2 + chalf;
      if (part < p.n_part && row_ok)
        p.partials[static_cast<size_t>(row) * p.part_stride + part] = make_float2(ssq, ssk);
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    // a wait gave up: give any copy still in flight (possibly signalling the peer) time to land
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, 1);
}

// ---------------------------------------------------------------- weight packing
__global__ void transpose_w_kernel(const uint8_t* __restrict__ w, uint8_t* __restrict__ wt, int H,
                                   int I) {
  __shared__ uint8_t tile[64][65];
  const int i0 = blockIdx.x * 64, h0 = blockIdx.y * 64;
  for (int r = threadIdx.y; r < 64; r += blockDim.y) {
    const int h = h0 + r, i = i0 + threadIdx.x;
    if (h < H && i < I) tile[r][threadIdx.x] = w[static_cast<size_t>(h) * I + i];
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 64; r += blockDim.y) {
    const int i = i0 + r, h = h0 + threadIdx.x;
    if (i < I && h < H) wt[static_cast<size_t>(i) * H + h] = tile[threadIdx.x][r];
  }
}

// Scale image of one (column tile, K stage), 4 KB: 128 rows (TMEM lanes) of 32
// bytes, stored as core matrices of 8 rows x 16 bytes, (row group, half) at
// (2 * group + half) * 128.  Row L, word c (0..7), byte j holds the exponent of
// column c * 32 + L % 32 of the tile and 32-block j of the stage, so that one
// tcgen05.cp 128x256b gives "TMEM lane n % 32 (in each lane quadrant), column n / 32,
// byte = block", the layout the block-scaled MMA reads.
__global__ void pack_sf_kernel(const uint8_t* __restrict__ e, uint8_t* __restrict__ sf, int H, int I,
                               int num_n, int num_k) {
  const size_t total = static_cast<size_t>(num_n) * num_k * SF_BYTES;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int off = static_cast<int>(idx % SF_BYTES);
    const size_t t = idx / SF_BYTES;
    const int kb = static_cast<int>(t % num_k);
    const int nt = static_cast<int>(t / num_k);
    // core matrices of 8 rows x 16 bytes: (row group rg, column half ch) at (2 rg + ch) * 128;
    // row L (TMEM lane), word cc (column), byte j (K block): column cc * 32 + L % 32
    const int cm = off / 128, within = off % 128;
    const int L = (cm / 2) * 8 + within / 16, cc = (cm % 2) * 4 + (within % 16) / 4, j = within % 4;
    const int nl = cc * 32 + L % 32;
    const int n = nt * BN + nl;
    const int hb = kb * (BK / 32) + j;
    uint8_t v = 127;
    if (nl < BN && n < I && hb < H / 32) v = e[static_cast<size_t>(hb) * I + n];
    sf[idx] = v;
  }
}

bool make_tmap_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                  uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};  // bytes per row (1-byte elements)
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t packed_sf_offset(int64_t H, int64_t I) {
  return ((static_cast<size_t>(H) * I + 1023) / 1024) * 1024;
}

size_t packed_weight_bytes(int64_t H, int64_t I) {
  const size_t num_n = (I + BN - 1) / BN, num_k = (H + BK - 1) / BK;
  return packed_sf_offset(H, I) + num_n * num_k * SF_BYTES;
}

cudaError_t launch_pack_weight(const uint8_t* w, const uint8_t* w_block_exp, int64_t H, int64_t I,
                               uint8_t* packed, cudaStream_t stream) {
  dim3 tb(64, 4), tg(static_cast<unsigned>((I + 63) / 64), static_cast<unsigned>((H + 63) / 64));
  transpose_w_kernel<<<tg, tb, 0, stream>>>(w, packed, static_cast<int>(H), static_cast<int>(I));
  const int num_n = static_cast<int>((I + BN - 1) / BN), num_k = static_cast<int>((H + BK - 1) / BK);
  const size_t total = static_cast<size_t>(num_n) * num_k * SF_BYTES;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((total + 255) / 256, 65535));
  pack_sf_kernel<<<blocks, 256, 0, stream>>>(w_block_exp, packed + packed_sf_offset(H, I),
                                             static_cast<int>(H), static_cast<int>(I), num_n, num_k);
  return cudaGetLastError();
}

cudaError_t launch_qkv_project(const ProjLaunch& L, cudaStream_t stream, const char** why) {
  Params p{};
  const int num_n = static_cast<int>((L.I + BN - 1) / BN), num_k = static_cast<int>(L.H / BK);
  const uint64_t sf_rows = static_cast<uint64_t>(num_n) * num_k * (SF_BYTES / 256);
  if (!make_tmap_2d(&p.tmap_a, L.a, L.H, L.T, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&p.tmap_b, L.w_t, L.H, L.I, BK, BN_HALF, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&p.tmap_sf, L.sf, 256, sf_rows, 256, 16, CU_TENSOR_MAP_SWIZZLE_NONE)) {
    *why = "cuTensorMapEncodeTiled failed or is unavailable";
    return cudaErrorInvalidValue;
  }
  p.a_scale = L.a_scale;
  p.wch = L.weight_scales;
  p.bias = L.bias;
  p.out = L.out;
  p.exps = L.exps;
  p.partials = L.partials;
  p.status = L.status;
  p.T = static_cast<int32_t>(L.T);
  p.I = static_cast<int32_t>(L.I);
  p.num_k = num_k;
  p.num_m = static_cast<int32_t>((L.T + PAIR_M - 1) / PAIR_M);
  p.num_n = num_n;
  p.q_end = L.q_end;
  p.k_end = L.k_end;
  p.n_part = L.n_part_tiles;
  p.n_exp = L.n_exp_blocks;
  p.part_stride = L.part_stride;
  p.exp_stride = L.exp_stride;
  p.s_begin = L.s_begin;
  p.s_end = L.s_end;
  p.q_gamma = L.q_gamma;
  p.k_gamma = L.k_gamma;
  p.wait_ns = static_cast<uint64_t>(L.wait_ns);
  p.stall_loads = L.stall_loads;
  p.head_dim = L.head_dim;
  p.nbsd = L.nbsd;
  p.out32 = (reinterpret_cast<uintptr_t>(L.out) & 31u) == 0;
  p.ph_begin = L.ph_begin;
  p.ph_end = L.ph_end;
  p.ph_carry = L.ph_carry;
  p.ph_q_gamma = L.ph_q_gamma;
  p.ph_k_gamma = L.ph_k_gamma;
  p.eps = L.eps;

  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    for (auto k : {qkv_project_kernel<0>, qkv_project_kernel<64>, qkv_project_kernel<128>})
      if (attr_err == cudaSuccess)
        attr_err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  });
  if (attr_err != cudaSuccess) {
    *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return attr_err;
  }
  const int num_tiles = p.num_m * p.num_n;
  const int pairs = std::max(1, std::min(num_tiles, device_sm_count() / 2));
  if (p.ph_end <= p.ph_begin)
    qkv_project_kernel<0><<<2 * pairs, NUM_THREADS, SMEM_ALLOC, stream>>>(p);
  else if (p.head_dim == 128)
    qkv_project_kernel<128><<<2 * pairs, NUM_THREADS, SMEM_ALLOC, stream>>>(p);
  else
    qkv_project_kernel<64><<<2 * pairs, NUM_THREADS, SMEM_ALLOC, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ra
