// Inline-PTX wrappers for the sm_103a tensor-core path: mbarriers (with bounded waits), TMA and
// bulk copies, tcgen05 MMA / TMEM loads and stores. Only the prefill GEMM includes this header.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace ds4 {
namespace tc {

// A wait that has not completed after this many SM cycles (about a second) is abandoned: the
// kernel records an error bit and stops instead of spinning forever. (A launch may set a shorter
// limit: see GemmArgs::timeout_cycles.)
constexpr long long kTimeoutCycles = 2000000000ll;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that may suspend the thread in hardware until the phase completes (or about 0.1 ms
// pass): a waiting warp takes no issue slots from the warps that have work.
__device__ __forceinline__ bool mbar_try_sleep(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}

// Waits for the phase of the given parity. Returns false (and raises the CTA's abort flag, error
// bit 2 of *err and bit 16 + site, which names the wait that gave up) if it does not complete in
// time, or if another thread already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag, int* err,
                                          int site = 0, long long limit = kTimeoutCycles) {
  if (mbar_try(b, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_sleep(b, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(err, 4 | (1 << (16 + site)));
      return false;
    }
  }
  return true;
}

// 2D tiled TMA load (box defined by the tensor map) completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::
          "r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}
// The same load multicast to every CTA of the cluster named in mask: the box lands at the same
// shared-memory offset in each, and each CTA's mbarrier at bar's offset receives the bytes.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;\n" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar)), "h"(mask)
      : "memory");
}

// Brings a tensor map's descriptor into the TMA unit's cache before its first use.
__device__ __forceinline__ void tmap_prefetch(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// Barrier over every thread of every CTA of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}

// ---- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(slot)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// tcgen05.commit (arrives on the mbarrier once all MMAs the thread issued before it have
// completed) by one lane that elect.sync picks, called by the whole converged warp: with all 32
// lanes active the elected lane is the same at every call, so it tracks that lane's MMAs.
__device__ __forceinline__ void tc_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(su32(bar))
      : "memory");
}

// Stores 32 consecutive 32-bit columns for each of the 32 lanes of the warp's TMEM lane quadrant
// (lane i of the warp writes TMEM lane quadrant_base + i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Eight MMAs of one 128-k stage (A in tensor memory, 64 columns from a_tmem; B as two 64-k
// sub-tiles with descriptors b0 and b1, each advanced 32 bytes per 16 k), issued by one elected
// lane of the converged warp: one elect and no compiler ordering between the eight. The first
// MMA accumulates into D only if accumulate != 0; the other seven always do.
__device__ __forceinline__ void tc_mma8_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0, uint64_t b1,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, t, e;\n .reg .b32 a;\n .reg .b64 b;\n"
      " setp.ne.b32 p, %5, 0;\n setp.eq.b32 t, %5, %5;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n"
      " add.u32 a, %1, 8;\n add.u64 b, %2, 2;\n @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, t;\n"
      " add.u32 a, %1, 16;\n add.u64 b, %2, 4;\n @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, t;\n"
      " add.u32 a, %1, 24;\n add.u64 b, %2, 6;\n @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, t;\n"
      " add.u32 a, %1, 32;\n @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], %3, %4, t;\n"
      " add.u32 a, %1, 40;\n add.u64 b, %3, 2;\n @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, t;\n"
      " add.u32 a, %1, 48;\n add.u64 b, %3, 4;\n @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, t;\n"
      " add.u32 a, %1, 56;\n add.u64 b, %3, 6;\n @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, t;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b0), "l"(b1), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The commits that release a stage: a multicast commit to the activation stage's barrier in every
// CTA of the cluster in mask (or a plain one if mask is 0) and a commit to the local A stage's
// barrier, issued by one elected lane.
__device__ __forceinline__ void tc_commit2_elect(uint64_t* b_bar, uint16_t mask, uint64_t* a_bar) {
  if (mask)
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%2];\n}\n" ::"r"(su32(b_bar)),
        "h"(mask), "r"(su32(a_bar))
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n}\n" ::"r"(su32(b_bar)),
        "r"(su32(a_bar))
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns of the warp's TMEM lane quadrant.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major tile in the 128-byte swizzled canonical layout:
// rows of 128 bytes (64 fp16 of K), 8-row atoms of 1024 bytes stacked along M/N.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);  // start address / 16
  d |= (uint64_t)1 << 16;                       // leading byte offset (unused by this layout)
  d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset: one 8-row atom
  d |= (uint64_t)1 << 46;                       // descriptor version
  d |= (uint64_t)2 << 61;                       // swizzle mode: 128 bytes
  return d;
}

// Instruction descriptor of kind::f16: fp16 A and B (both K-major), fp32 accumulator, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}
// Named barrier that also returns the AND of a predicate over its threads: every participant
// gets the same answer (so a group decides together whether to enter code with more barriers).
__device__ __forceinline__ bool named_bar_all(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, %2, %3, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

}  // namespace tc
}  // namespace ds4
