// Inline-PTX helpers for sm_103a: mbarriers, TMA (cp.async.bulk), and the
// 5th-generation tensor core (tcgen05: TMEM allocation, MMA, copies, loads).
// Each wrapper is written from the PTX ISA.  Most are one instruction; the MMA
// stage helpers issue a whole pipeline stage (or two) from one asm block, for the
// reason given at tc_mma_stage_pair_mxf8.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace ra {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// adds `bytes` to the transaction count of the current phase without arriving
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// true once the phase with the given parity has completed
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded mbarrier waits (limit in ns of %globaltimer).  A wait gives up when
// the limit passes or when *abort_flag is set, and then sets *abort_flag.
// single thread:
__device__ inline bool bounded_wait_one(uint32_t bar, uint32_t parity, uint64_t limit,
                                        volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*abort_flag || globaltimer_ns() - t0 > limit) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}
// whole warp (every lane returns the same answer):
__device__ inline bool bounded_wait_warp(uint32_t bar, uint32_t parity, uint64_t limit,
                                         volatile int* abort_flag) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((i & 31u) == 31u) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0) {
        const uint64_t t = globaltimer_ns();
        if (t0 == 0) t0 = t;
        else if (*abort_flag || t - t0 > limit) give_up = 1;
      }
      give_up = __shfl_sync(0xffffffffu, give_up, 0);
      if (give_up) {
        if ((threadIdx.x & 31) == 0) *abort_flag = 1;
        return false;
      }
    }
  }
}
// used while leaving: wait for the phase, at most `limit` ns; false if it did not complete
__device__ inline bool bounded_drain(uint32_t bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA / bulk copies
__device__ __forceinline__ void prefetch_tensormap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// plain bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// plain bulk copy shared -> global, tracked by the issuing thread's bulk groups;
// both addresses 16-byte aligned, bytes % 16 == 0
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N of this thread's bulk groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until every bulk group of this thread has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in bits
// [0,14), leading byte offset >> 4 in [16,30), stride byte offset >> 4 in
// [32,46), version 1 in [46,48), base offset 0, layout type in [61,64).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                          uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}
constexpr uint32_t kLayoutNone = 0;
constexpr uint32_t kLayoutSwizzle128B = 2;

// K-major operand tile written by TMA with 128-byte swizzle: rows of 128 bytes,
// 8-row (1024-byte) swizzle atoms stacked along M/N.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  return sdesc(saddr, 16, 1024, kLayoutSwizzle128B);
}
// 32 rows x 16 bytes, rows contiguous (8-row core matrices 128 bytes apart)
__device__ __forceinline__ uint64_t sdesc_scale_rows(uint32_t saddr) {
  return sdesc(saddr, 0, 128, kLayoutNone);
}
// 128 rows x 32 bytes in core matrices of 8 rows x 16 bytes: (row group rg, half ch)
// at (2 rg + ch) * 128 bytes, i.e. 128 bytes between the halves, 256 between row groups
__device__ __forceinline__ uint64_t sdesc_scale_image(uint32_t saddr) {
  return sdesc(saddr, 128, 256, kLayoutNone);
}

// ---------------------------------------------------------------- clusters and CTA pairs
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// arrive on an mbarrier of any CTA of the cluster (a shared::cluster address) without
// release semantics: it does not wait for this thread's earlier memory writes to
// become visible to the cluster
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// TMA tile load whose completion may be signalled on the peer CTA's mbarrier
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// arrive on the mbarrier at `bar` in every CTA of `cta_mask` once this thread's
// tcgen05 ops have completed
__device__ __forceinline__ void tc_commit_pair_multicast(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// True once both mbarriers at bar0 and bar0 + 8 have completed the phase with the
// given parity.  The two non-blocking probes go out back to back, so one
// shared-memory round trip answers both.
__device__ __forceinline__ bool mbar_test_wait_pair(uint32_t bar0, uint32_t parity) {
  uint32_t both;
  asm volatile(
      "{\n\t"
      ".reg .pred f0, f1;\n\t"
      ".reg .b32 bar1;\n\t"
      "add.u32 bar1, %1, 8;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 f0, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 f1, [bar1], %2;\n\t"
      "and.pred f0, f0, f1;\n\t"
      "selp.u32 %0, 1, 0, f0;\n\t"
      "}"
      : "=r"(both)
      : "r"(bar0), "r"(parity)
      : "memory");
  return both != 0;
}

// One pipeline stage of the 2-SM block-scaled MMA from one asm block, with a
// look-ahead probe of the next stage's full barrier: probe nbar for phase parity
// nphase (mbarrier.test_wait, acquire), copy the stage's W scale image into the TMEM
// slot sfb, issue four K=32 MMAs into d (the first accumulates only when
// acc_first != 0), commit to the stage's empty barrier ebar in both CTAs, and only
// then read the probe's predicate (see tc_mma_stage_pair_mxf8 below for why the read
// comes last).  For calls whose number of K steps is odd.
__device__ __forceinline__ bool tc_mma_stage_mxf8(uint32_t nbar, uint32_t nphase, uint32_t sfb, uint64_t sfd,
                                                  uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc,
                                                  uint32_t sfa, uint32_t acc_first, uint32_t ebar) {
  uint32_t full;
  asm volatile(
      "{\n\t"
      ".reg .pred full0, acc0, on;\n\t"
      ".reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      ".reg .b32 id1, id2, id3;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 full0, [%1], %2;\n\t"
      "or.b32 id1, %8, 0x20000010;\n\t"
      "or.b32 id2, %8, 0x40000020;\n\t"
      "or.b32 id3, %8, 0x60000030;\n\t"
      "setp.ne.b32 acc0, %10, 0;\n\t"
      "setp.eq.b32 on, 0, 0;\n\t"
      "add.s64 a1, %6, 2;\n\tadd.s64 b1, %7, 2;\n\t"
      "add.s64 a2, %6, 4;\n\tadd.s64 b2, %7, 4;\n\t"
      "add.s64 a3, %6, 6;\n\tadd.s64 b3, %7, 6;\n\t"
      "tcgen05.cp.cta_group::2.128x256b [%3], %4;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], %6, %7, %8, [%9], [%3], acc0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a1, b1, id1, [%9], [%3], on;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a2, b2, id2, [%9], [%3], on;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a3, b3, id3, [%9], [%3], on;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%11], %12;\n\t"
      "selp.u32 %0, 1, 0, full0;\n\t"
      "}"
      : "=r"(full)
      : "r"(nbar), "r"(nphase), "r"(sfb), "l"(sfd), "r"(d), "l"(ad), "l"(bd), "r"(idesc), "r"(sfa),
        "r"(acc_first), "r"(ebar), "h"(static_cast<uint16_t>(0x3))
      : "memory");
  return full != 0;
}

// Two consecutive pipeline stages of the 2-SM block-scaled MMA, issued from one asm
// block, with a look-ahead probe of the next two stages' full barriers.
//
// For each of the two stages: copy the stage's W scale image into its TMEM slot
// (sfb0, then sfb0 + 8), issue four K=32 MMAs into the accumulator d (the first one
// of the pair accumulates only when acc_first != 0), and commit to the stage's empty
// barrier in both CTAs (ebar0, then ebar0 + 8).  The second stage's operands sit one
// stage further in shared memory: +1024 in the descriptors' 16-byte address units
// for 16 KB operand stages, +256 for the 4 KB scale images.
//
// Before any of that, mbarrier.test_wait (acquire) probes the full barriers nbar0 and
// nbar0 + 8 for phase parity nphase; the result (both complete) is returned.  Its
// predicate is read only after the last commit.  A shared-memory round trip of the
// issuing thread takes hundreds of cycles while the tensor core streams operands,
// and the thread cannot issue past an instruction that waits for such a result; with
// the read at the end, the probe's latency overlaps the issue of eight MMAs instead
// of leaving the tensor pipe without queued work (measured: 27.8k cycles per
// 160-MMA tile with a wait per stage, 20.5k with this form, 20.48k ideal).
// The caller keeps the ring and the scale slots from wrapping inside a pair (even
// first stage, even ring length).
__device__ __forceinline__ bool tc_mma_stage_pair_mxf8(uint32_t nbar0, uint32_t nphase, uint32_t sfb0,
                                                       uint64_t sfd0, uint32_t d, uint64_t ad0, uint64_t bd0,
                                                       uint32_t idesc, uint32_t sfa, uint32_t acc_first,
                                                       uint32_t ebar0) {
  uint32_t both_full;
  asm volatile(
      "{\n\t"
      ".reg .pred full0, full1, acc0, on;\n\t"
      ".reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7, sfd1;\n\t"
      ".reg .b32 id1, id2, id3, sfb1, nbar1, ebar1;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 full0, [%1], %2;\n\t"
      "add.u32 nbar1, %1, 8;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 full1, [nbar1], %2;\n\t"
      // the scale-factor ids of K steps 1..3 (bits [29,31) for A, [4,6) for B)
      "or.b32 id1, %8, 0x20000010;\n\t"
      "or.b32 id2, %8, 0x40000020;\n\t"
      "or.b32 id3, %8, 0x60000030;\n\t"
      "setp.ne.b32 acc0, %10, 0;\n\t"
      "setp.eq.b32 on, 0, 0;\n\t"
      "add.s64 a1, %6, 2;\n\tadd.s64 b1, %7, 2;\n\t"
      "add.s64 a2, %6, 4;\n\tadd.s64 b2, %7, 4;\n\t"
      "add.s64 a3, %6, 6;\n\tadd.s64 b3, %7, 6;\n\t"
      "tcgen05.cp.cta_group::2.128x256b [%3], %4;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], %6, %7, %8, [%9], [%3], acc0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a1, b1, id1, [%9], [%3], on;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a2, b2, id2, [%9], [%3], on;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a3, b3, id3, [%9], [%3], on;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%11], %12;\n\t"
      "add.u32 sfb1, %3, 8;\n\tadd.s64 sfd1, %4, 256;\n\t"
      "add.s64 a4, %6, 1024;\n\tadd.s64 b4, %7, 1024;\n\t"
      "add.s64 a5, %6, 1026;\n\tadd.s64 b5, %7, 1026;\n\t"
      "add.s64 a6, %6, 1028;\n\tadd.s64 b6, %7, 1028;\n\t"
      "add.s64 a7, %6, 1030;\n\tadd.s64 b7, %7, 1030;\n\t"
      "add.u32 ebar1, %11, 8;\n\t"
      "tcgen05.cp.cta_group::2.128x256b [sfb1], sfd1;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a4, b4, %8, [%9], [sfb1], on;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a5, b5, id1, [%9], [sfb1], on;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a6, b6, id2, [%9], [sfb1], on;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%5], a7, b7, id3, [%9], [sfb1], on;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [ebar1], %12;\n\t"
      "and.pred full0, full0, full1;\n\t"
      "selp.u32 %0, 1, 0, full0;\n\t"
      "}"
      : "=r"(both_full)
      : "r"(nbar0), "r"(nphase), "r"(sfb0), "l"(sfd0), "r"(d), "l"(ad0), "l"(bd0), "r"(idesc), "r"(sfa),
        "r"(acc_first), "r"(ebar0), "h"(static_cast<uint16_t>(0x3))
      : "memory");
  return both_full != 0;
}

// ---------------------------------------------------------------- small utils
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// 2^k as a float for |k| <= 126, built from the exponent field
__device__ __forceinline__ float exp2_int(int k) { return __uint_as_float(static_cast<uint32_t>(127 + k) << 23); }
// e such that x * 2^-e < 2^15 with x's leading bit at 2^14 (x >= 0 finite); clamped to [-100, 100]
__device__ __forceinline__ int scale_exponent(float x) {
  const int be = static_cast<int>((__float_as_uint(x) >> 23) & 0xFFu);  // biased exponent, floor(log2 x) + 127
  int e = be == 0 ? -100 : be - 127 - 14;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) { return make_float2(bf16_lo(v), bf16_hi(v)); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace ra
