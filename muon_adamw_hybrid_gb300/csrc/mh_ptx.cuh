// Inline-PTX helpers for sm_103a: mbarriers, TMA tensor loads, tcgen05 MMA /
// TMEM, with bounded waits. Everything here is device code written against
// the public PTX ISA (mbarrier, cp.async.bulk.tensor, tcgen05.*).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace mh {

// Device status codes written to the workspace status word.
enum : int {
  DEV_OK = 0,
  DEV_TIMEOUT_TMA = 1,      // a GEMM producer waited too long for a free stage
  DEV_TIMEOUT_MMA = 2,      // a GEMM MMA issuer waited too long for operands / accumulators
  DEV_TIMEOUT_EPI = 3,      // a GEMM epilogue waited too long for an accumulator
  DEV_TIMEOUT_STREAM = 4    // a streaming elementwise pass waited too long for a stage
};

// A bounded wait gives up after this many SM clock cycles (about 1 s at the
// GB300's clocks) unless the launch sets its own limit; no legitimate wait in
// these kernels is longer than a few milliseconds. Draining after an abort
// always uses kDrainLimitCycles, so that copies and MMAs already issued land
// before a CTA leaves, however short the launch's own limit is.
constexpr long long kWaitLimitCycles = 2000000000LL;
constexpr long long kDrainLimitCycles = kWaitLimitCycles / 4;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, with acquire semantics at cluster scope: for a phase
// completed by an arrive from the other CTA of the cluster, after which this
// thread reads data that CTA stored into this CTA's shared memory.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Returns false if the
// CTA-wide abort flag is raised, or if the wait exceeds `limit` cycles, in
// which case it raises the abort flag and records `code` in the status word.
// CLUSTER: acquire at cluster scope (see mbar_try_wait_cluster).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, int* status,
                                                  int code, long long limit) {
  const uint32_t addr = smem_addr(bar);
  auto poll = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(addr, parity) : mbar_try_wait(addr, parity);
  };
  if (poll()) return true;
  const long long t0 = clock64();
  // The abort flag and the clock are checked every 32 unsuccessful polls, so
  // that a waiting thread notices the phase as soon as it completes. try_wait
  // may suspend the thread for a while on each poll, so under a limit
  // shortened below the default they are checked after every poll instead.
  const int polls = limit < kWaitLimitCycles ? 1 : 32;
  while (true) {
#pragma unroll 1
    for (int i = 0; i < polls; ++i)
      if (poll()) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicCAS(status, DEV_OK, code);
      return false;
    }
  }
}

// Bounded wait used only while draining after an abort (kDrainLimitCycles).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_addr(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(addr, parity)) {
    if (clock64() - t0 > kDrainLimitCycles) return;
  }
}

// Shared-memory address of the same offset as `local` in CTA `cta` of the
// cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* local, uint32_t cta) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote)
               : "r"(smem_addr(local)), "r"(cta));
  return remote;
}

// Arrives once on the mbarrier at the offset of `local_bar` in CTA `cta` of
// the cluster, releasing this thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* local_bar, uint32_t cta) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   cluster_map(local_bar, cta))
               : "memory");
}

// As mbar_arrive_cluster without release semantics: the arrive orders none of
// this thread's earlier writes (it does not wait for them to be performed).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint64_t* local_bar, uint32_t cta) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   cluster_map(local_bar, cta))
               : "memory");
}

// Arrives once on an mbarrier of this CTA without release semantics.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Loads a 32-bit word of this CTA's shared memory with acquire semantics at
// CTA scope: no later memory operation of this thread is performed before it.
__device__ __forceinline__ uint32_t ld_acquire_cta_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p))
               : "memory");
  return v;
}

// Loads a 32-bit word of this CTA's shared memory with acquire semantics at
// cluster scope: no later memory operation of this thread is performed before
// it.
__device__ __forceinline__ uint32_t ld_acquire_cluster_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.acquire.cluster.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p))
               : "memory");
  return v;
}

// Arrives once on the mbarrier at the offset of `local_bar` in CTA `cta` of
// the cluster and adds `bytes` to the transaction count its current phase
// waits for; relaxed: no earlier write of this thread is ordered by it.
__device__ __forceinline__ void mbar_arrive_expect_tx_relaxed(uint64_t* local_bar, uint32_t cta,
                                                              uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
          cluster_map(local_bar, cta)),
      "r"(bytes)
      : "memory");
}

// Asynchronous store of `v` to the 32-bit word at the offset of `local` in
// CTA `cta` of the cluster (this CTA included); its completion counts 4
// bytes of transactions on the mbarrier at the offset of `local_bar` in that
// CTA, so a thread that sees the barrier's phase complete sees the value.
__device__ __forceinline__ void st_async_u32(const void* local, uint32_t cta, uint32_t v,
                                             uint64_t* local_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(
          cluster_map(local, cta)),
      "r"(v), "r"(cluster_map(local_bar, cta))
      : "memory");
}

// Stores `v` to the 32-bit word at the offset of `local` in CTA `cta` of the
// cluster.
__device__ __forceinline__ void st_cluster_u32(const void* local, uint32_t cta, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_map(local, cta)), "r"(v)
               : "memory");
}

// Adds `bytes` to the transaction count of the mbarrier's current phase
// without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Arrives on `bar` once every cp.async this thread issued so far has landed.
// The arrival is not counted in advance (.noinc): the barrier's expected
// count includes it.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 3-D tiled TMA load into CTA shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Same, multicast to every CTA of the cluster in `mask`: the data lands at the
// same shared-memory offset in each of them and completes bytes on the
// mbarrier at the same offset in each.
__device__ __forceinline__ void tma_load_3d_mc(void* smem_dst, const void* tmap, uint64_t* bar,
                                               int32_t c0, int32_t c1, int32_t c2, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2),
      "h"(mask)
      : "memory");
}

// 3-D tiled TMA store from CTA shared memory, tracked by the issuing thread's
// bulk async-groups. Elements of the box outside the tensor map's extents are
// not written.
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* smem_src, int32_t c0,
                                             int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(smem_addr(smem_src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N of this thread's committed bulk groups still read
// their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until all of this thread's committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Orders this thread's earlier shared-memory writes before later accesses of
// the async proxy (a TMA store reading them).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Writes `v` to the int at the same shared-memory offset as `local` in CTA
// `cta` of the cluster.
__device__ __forceinline__ void st_cluster_s32(volatile int* local, uint32_t cta, int v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote)
               : "r"(smem_addr(const_cast<int*>(local))), "r"(cta));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---- tcgen05 ----------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
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

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// As tc_commit, arriving on the mbarrier at the same offset in every CTA of
// the cluster in `mask`.
__device__ __forceinline__ void tc_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// Warp-collective load of 32 lanes x 32 consecutive fp32 columns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
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

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D.
// a_mn / b_mn: 0 = K-major operand, 1 = MN-major operand.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                                  // D format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | (static_cast<uint32_t>(a_mn) << 15)      // A major
         | (static_cast<uint32_t>(b_mn) << 16)      // B major
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

}  // namespace mh
