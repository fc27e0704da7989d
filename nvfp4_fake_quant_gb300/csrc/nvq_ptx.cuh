// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tensor loads, tcgen05 (TMEM allocation, UMMA issue, commit, TMEM loads) and
// the shared-memory / instruction descriptors of kind::f16 UMMAs.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace nvq {

// Code a kernel records in the device error word (read and cleared by
// nvq_device_status) when one of its bounded waits ran out.
enum : int { kErrTimeout = 5 };

// Limit of one bounded wait.  Waits in a correct kernel last microseconds.
#ifndef NVQ_WAIT_LIMIT_NS
#define NVQ_WAIT_LIMIT_NS 2000000000ull
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// `limit_ns` (setting *abort, which the kernel turns into kErrTimeout in the
// device error word when it leaves) or as soon as another thread of the block
// has set *abort.  Returns true on success.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = NVQ_WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        if (abort != nullptr) *abort = 1;
        return false;
      }
    }
  }
}

// mbar_wait by every lane of a warp with a warp-uniform result, so that the
// .sync.aligned tcgen05 instructions that follow run on a converged warp even
// when some lane's wait gave up.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint64_t limit_ns = NVQ_WAIT_LIMIT_NS) {
  const bool ok = mbar_wait(bar, parity, abort, limit_ns);
  return __all_sync(0xFFFFFFFFu, ok);
}

// One arrival per warp: every lane's prior writes and fences are ordered before
// lane 0's arrive by the warp barrier.  Barriers fed this way count warps.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Block teardown: report an aborted wait in the device error word.
__device__ __forceinline__ void report_abort(volatile int* abort, int* err) {
  if (threadIdx.x == 0 && *abort) atomicExch(err, kErrTimeout);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Warp-collective forms (see "warp-collective issue" below): every lane calls
// with the same arguments, one elected lane issues.
__device__ __forceinline__ void mbar_arrive_expect_tx_w(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_w(void* smem_dst, const CUtensorMap* map, int c0, int c1,
                                              int c2, int c3, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

// Contiguous copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to shared memory, completing on `bar` (tx bytes).  Warp-collective.
__device__ __forceinline__ void bulk_load_w(void* smem_dst, const void* src, uint32_t bytes,
                                            uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      "\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster (arrive has release, wait acquire
// semantics): orders barrier initialisation before any remote arrival and keeps
// a CTA's shared memory alive until its peers are done with it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// 4-D tiled load written to the same shared-memory offset in every CTA of
// `mask` (cluster ranks), each completing `bytes` of tx on the mbarrier at
// bar's offset in that CTA.  Warp-collective (one elected lane issues).
__device__ __forceinline__ void tma_load_4d_mc_w(void* smem_dst, const CUtensorMap* map, int c0,
                                                 int c1, int c2, int c3, uint64_t* bar,
                                                 uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3, %4, %5}], [%6], %7;\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}
// Contiguous copy (size % 16 == 0, 16-byte aligned) to the same offset in every
// CTA of `mask`.  Warp-collective.
__device__ __forceinline__ void bulk_load_mc_w(void* smem_dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1], %2, [%3], %4;\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

// --------------------------------------------------------------- TMA store
// 4-D tiled store of a shared-memory box (written by this thread's proxy-fenced
// stores) into global memory; elements outside the tensor are not written.
// Issued, committed and waited on by one thread (bulk groups are per thread).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* smem_src, int c0,
                                             int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(smem_src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N of this thread's committed bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ tcgen05
// TMEM allocation (one warp, .sync.aligned): writes the base address to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// --------------------------------------------------- warp-collective issue
// Called by every lane of a converged warp with the same arguments; elect.sync
// inside the asm block picks the one lane that issues.  Keeping the issuing
// warp converged lets the compiler keep descriptors and addresses in
// warp-uniform registers: issuing from one lane of a divergent branch costs
// about 65 cycles per tcgen05.mma, more than a 128x64x16 UMMA takes to run.
//
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (f16 or bf16 inputs, f32 accumulate).
__device__ __forceinline__ void umma_f16_ss_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same with A read from TMEM: a_tmem addresses lane 0 of the 128 x 16 A slice,
// stored as 8 consecutive 32-bit columns of two 16-bit elements each (element
// 2c in the low half of column c).  B and the instruction descriptor as above.
__device__ __forceinline__ void umma_f16_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on `bar` when every tcgen05 op the issuing thread has issued so
// far is done.
__device__ __forceinline__ void umma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// umma_commit_w, arriving on the mbarrier at bar's offset in every CTA of `mask`.
__device__ __forceinline__ void umma_commit_mc_w(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// ------------------------------------------- grouped issue with commits
// A group of UMMAs and the tcgen05.commit(s) after them from one asm block and
// one elected lane, operands precomputed by the caller.  The issuing warps share
// their sub-partitions with busy elementwise warps and get few issue slots, so
// every instruction between the barrier that releases a group and the UMMAs
// delays the UMMAs.  Commits go to the mbarrier at shared address c0 and, unless
// c1 is 0 (no barrier lives at shared address 0), to c1.
//
// kSteps (4 or 8) kind::f16 UMMAs into one accumulator, A and B from
// shared-memory descriptors: the first with the given accumulate flag, the rest
// accumulating.
template <int kSteps>
__device__ __forceinline__ void umma_f16_group_w(uint32_t d, const uint64_t* ad, const uint64_t* bd,
                                                 uint32_t idesc, uint32_t acc, uint32_t c0,
                                                 uint32_t c1) {
  static_assert(kSteps == 4 || kSteps == 8, "4 or 8 K steps");
  if constexpr (kSteps == 8) {
    asm volatile(
        "{\n\t.reg .pred p, e, t, q;\n\t"
        "setp.ne.b32 p, %2, 0;\n\t"
        "setp.eq.u32 t, 0, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.and.u32 q, %20, 0, e;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %1, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %17, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %10, %18, %1, t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%19];\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%20];\n\t}"
        ::"r"(d), "r"(idesc), "r"(acc), "l"(ad[0]), "l"(ad[1]), "l"(ad[2]), "l"(ad[3]),
        "l"(ad[4]), "l"(ad[5]), "l"(ad[6]), "l"(ad[7]), "l"(bd[0]), "l"(bd[1]), "l"(bd[2]),
        "l"(bd[3]), "l"(bd[4]), "l"(bd[5]), "l"(bd[6]), "l"(bd[7]), "r"(c0), "r"(c1)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, e, t, q;\n\t"
        "setp.ne.b32 p, %2, 0;\n\t"
        "setp.eq.u32 t, 0, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.and.u32 q, %12, 0, e;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %1, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %9, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %10, %1, t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11];\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%12];\n\t}"
        ::"r"(d), "r"(idesc), "r"(acc), "l"(ad[0]), "l"(ad[1]), "l"(ad[2]), "l"(ad[3]),
        "l"(bd[0]), "l"(bd[1]), "l"(bd[2]), "l"(bd[3]), "r"(c0), "r"(c1)
        : "memory");
  }
}

// kSteps (1 or 2) block-scaled kind::mxf4nvf4 UMMAs (K = 64 each) starting a
// fresh accumulator; sa/sb: TMEM addresses of the scale operands of the first K
// step (the next step's are 4 columns on).
template <int kSteps>
__device__ __forceinline__ void umma_fp4_group_w(uint32_t d, const uint64_t* ad, const uint64_t* bd,
                                                 uint32_t idesc, uint32_t sa, uint32_t sb,
                                                 uint32_t c0, uint32_t c1) {
  static_assert(kSteps == 1 || kSteps == 2, "D = 64 or 128");
  if constexpr (kSteps == 2) {
    asm volatile(
        "{\n\t.reg .pred e, t, f, q;\n\t.reg .b32 sa1, sb1;\n\t"
        "setp.eq.u32 t, 0, 0;\n\t"
        "setp.ne.u32 f, 0, 0;\n\t"
        "add.u32 sa1, %4, 4;\n\t"
        "add.u32 sb1, %5, 4;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.and.u32 q, %9, 0, e;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %2, %6, %1, "
        "[%4], [%5], f;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %3, %7, %1, "
        "[sa1], [sb1], t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%8];\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%9];\n\t}"
        ::"r"(d), "r"(idesc), "l"(ad[0]), "l"(ad[1]), "r"(sa), "r"(sb), "l"(bd[0]), "l"(bd[1]),
        "r"(c0), "r"(c1)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, f, q;\n\t"
        "setp.ne.u32 f, 0, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.and.u32 q, %7, 0, e;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %2, %3, %1, "
        "[%4], [%5], f;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t}"
        ::"r"(d), "r"(idesc), "l"(ad[0]), "l"(bd[0]), "r"(sa), "r"(sb), "r"(c0), "r"(c1)
        : "memory");
  }
}

// Eight kind::f16 UMMAs (K = 16 each) into the accumulator d with A read from
// TMEM at a[k] and B through the descriptor b0 advanced by 2048 k bytes (128 k
// in its start-address field, which does not carry below 2^18 bytes of shared
// memory): an MN-major B whose K steps are 16 rows of 128 bytes.
__device__ __forceinline__ void umma_f16_ts8_w(uint32_t d, const uint32_t (&a)[8], uint64_t b0,
                                               uint32_t idesc, uint32_t acc, uint32_t c0,
                                               uint32_t c1) {
  asm volatile(
      "{\n\t.reg .pred p, e, t, q;\n\t.reg .b32 lo, hi;\n\t"
      ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      "setp.ne.b32 p, %2, 0;\n\t"
      "setp.eq.u32 t, 0, 0;\n\t"
      "mov.b64 {lo, hi}, %11;\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b1, {lo, hi};\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b2, {lo, hi};\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b3, {lo, hi};\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b4, {lo, hi};\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b5, {lo, hi};\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b6, {lo, hi};\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b7, {lo, hi};\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.and.u32 q, %13, 0, e;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %1, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], b1, %1, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], b2, %1, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], b3, %1, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], b4, %1, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], b5, %1, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], b6, %1, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%10], b7, %1, t;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%12];\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%13];\n\t}"
      ::"r"(d), "r"(idesc), "r"(acc), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]),
      "r"(a[5]), "r"(a[6]), "r"(a[7]), "l"(b0), "r"(c0), "r"(c1)
      : "memory");
}

// Four pairs of kind::f16 UMMAs with A in TMEM: pair k adds A at a[k] into d0
// and A at a[k] + 8 into d1, both with B through b0 advanced by 2048 k bytes;
// the first pair with the given accumulate flag.
__device__ __forceinline__ void umma_f16_ts4x2_w(uint32_t d0, uint32_t d1, const uint32_t (&a)[4],
                                                 uint64_t b0, uint32_t idesc, uint32_t acc,
                                                 uint32_t c0, uint32_t c1) {
  asm volatile(
      "{\n\t.reg .pred p, e, t, q;\n\t.reg .b32 lo, hi, a0, a1, a2, a3;\n\t"
      ".reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %3, 0;\n\t"
      "setp.eq.u32 t, 0, 0;\n\t"
      "mov.b64 {lo, hi}, %8;\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b1, {lo, hi};\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b2, {lo, hi};\n\t"
      "add.u32 lo, lo, 128;\n\tmov.b64 b3, {lo, hi};\n\t"
      "add.u32 a0, %4, 8;\n\tadd.u32 a1, %5, 8;\n\t"
      "add.u32 a2, %6, 8;\n\tadd.u32 a3, %7, 8;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.and.u32 q, %10, 0, e;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %2, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%1], [a0], %8, %2, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], b1, %2, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%1], [a1], b1, %2, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], b2, %2, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%1], [a2], b2, %2, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], b3, %2, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%1], [a3], b3, %2, t;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%9];\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n\t}"
      ::"r"(d0), "r"(d1), "r"(idesc), "r"(acc), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]),
      "l"(b0), "r"(c0), "r"(c1)
      : "memory");
}

// Shared-memory address of an mbarrier as a commit target (0: none).
__device__ __forceinline__ uint32_t bar_u32(uint64_t* bar) { return smem_u32(bar); }

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Store 16 consecutive 32-bit columns of this thread's lane (32x32b shape).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32); id 1..15.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
// Matrices are stored in 128-byte-swizzled atoms of 8 rows x 128 bytes,
// 1024-byte aligned, exactly as a TMA load with CU_TENSOR_MAP_SWIZZLE_128B
// writes them.
//   K-major operand (rows of the M/N dim, 64 K-elements per 128-byte row):
//     SBO = byte distance between consecutive groups of 8 rows; LBO unused.
//     Advancing K by 16 elements inside an atom adds 32 bytes to the start.
//   MN-major operand (rows of the K dim, 64 M/N-elements per 128-byte row):
//     LBO = byte distance between consecutive 64-element M/N chunks,
//     SBO = byte distance between consecutive groups of 8 K-rows.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version (Blackwell)
  d |= static_cast<uint64_t>(2) << 61;  // swizzle mode: 128-byte
  return d;
}

// Instruction descriptor of a kind::f16 UMMA with f32 accumulation.
//   ab_bf16: 1 = both operands bf16, 0 = both f16.  a_mn/b_mn: operand stored
//   MN-major (1) or K-major (0).  M in {64,128}, N % 16 == 0, N <= 256.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int ab_bf16, int a_mn, int b_mn) {
  return (1u << 4)                                  // D format: f32
         | (static_cast<uint32_t>(ab_bf16) << 7)    // A format
         | (static_cast<uint32_t>(ab_bf16) << 10)   // B format
         | (static_cast<uint32_t>(a_mn) << 15)      // A major
         | (static_cast<uint32_t>(b_mn) << 16)      // B major
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Shared-memory descriptor with an explicit layout type (bits 61-63):
// 0 = no swizzle (8-row x 16-byte core matrices), 2 = 128-byte, 4 = 64-byte,
// 6 = 32-byte swizzle.  For a K-major operand whose rows are `w` bytes wide and
// stored with the w-byte swizzle (as a TMA load with that swizzle and a box
// `w` bytes wide writes them), SBO = 8 * w and LBO is unused.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                          uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// Instruction descriptor of a block-scaled kind::mxf4nvf4 UMMA: A and B E2M1
// (format code 1), K-major, f32 accumulation, one unsigned E4M3 scale per 16
// K-elements (scale type bit 23 = 0), K = 64 per instruction (bit 31 = 0),
// scale-factor data ids 0.  M = 128, N % 8 == 0, N <= 256.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(int M, int N) {
  return (1u << 7)                                 // A format: E2M1
         | (1u << 10)                              // B format: E2M1
         | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// D[tmem] (+)= (A * sA) (B * sB)^T, E2M1 A and B in shared memory (K-major,
// two codes a byte, the even element in the low nibble), one E4M3 scale per
// 16 K-elements of each row read from TMEM at sfa_tmem / sfb_tmem.  K = 64.
__device__ __forceinline__ void umma_fp4_ss_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t sfa_tmem,
                                              uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Copy 32 rows x 16 bytes (512 contiguous bytes of shared memory, row r at
// 16 r) into TMEM columns [col, col + 4) of lanes r, r + 32, r + 64, r + 96
// (the same rows in each of the four lane quadrants).  Ordered before the
// tcgen05.mma instructions the same thread issues after it.
__device__ __forceinline__ void tmem_cp_32x128_x4_w(uint32_t taddr, uint32_t saddr) {
  const uint64_t d = sdesc(saddr, 128, 128, 0);
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(d)
      : "memory");
}

// Byte offset of element (row, col) of a 16-bit matrix stored as 128-byte
// swizzled atoms: 64 columns per atom column block of `rows_total` rows.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col, uint32_t rows_total) {
  const uint32_t blk = col >> 6;
  const uint32_t cc = col & 63u;
  const uint32_t chunk = (cc >> 3) ^ (row & 7u);
  return blk * rows_total * 128u + row * 128u + chunk * 16u + (cc & 7u) * 2u;
}

}  // namespace nvq
