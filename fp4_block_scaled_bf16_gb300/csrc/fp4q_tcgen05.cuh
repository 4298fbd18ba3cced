// fp4q_tcgen05.cuh -- PTX wrappers shared by the two GEMM kernels of
// libfp4q.so on sm_103a: bounded mbarrier waits with a CTA-wide abort flag,
// tcgen05 fences, TMEM allocation, MMA commits, TMEM loads, the K-major
// 128-byte-swizzled shared-memory matrix descriptor, 16-byte shared stores,
// and the cluster-pair primitives of the two-SM MMA.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp4q_device.cuh"
#include "fp4q_pipeline.cuh"

namespace fp4q {

// Bounded wait on the phase with the given parity.  False when the CTA's
// abort flag is set or the cycle budget runs out.  The first probe is inlined
// at the call site; only a wait that does not complete at once pays a call.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            long long budget) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) return false;
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          long long budget) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, budget);
}
__device__ __forceinline__ void fail(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  atomicOr(status, kStatusTimeout);
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// Waits for this thread's TMEM loads; the registers they wrote are then
// passed through empty statements that come after the wait, so that no use
// of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t* r, int n) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < n; ++i) asm volatile("" : "+r"(r[i]));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  tmem_ld_wait(r, 32);
}
// The same load without the wait: the caller calls tmem_ld_wait before
// reading r.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes (64 FP16, or 256 packed E2M1) grouped by 8 into 1024-byte atoms
// (stride-dimension offset 1024 B); the leading-dimension offset is unused in
// this mode.  Advancing the start address by 32 bytes moves one MMA K step
// along the row (K16 for FP16, K64 for E2M1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------- CTA pairs
// Wrappers for kernels launched in clusters of two that use the two-SM MMA
// (cta_group::2): the rank-0 CTA issues the MMAs, which read operands from
// both CTAs' shared memory and TMEM and write both CTAs' TMEM.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of both CTAs: release what this CTA wrote, acquire the peer's.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on the barrier at the same shared-memory offset in the rank-0 CTA.
// The arrival has the default semantics (release at CTA scope), as the
// vendor's own cluster pipelines use for remote arrivals.  What it publishes
// is work this CTA has finished on its own shared memory (stores fenced to
// the async proxy by every writing thread) or TMEM (tcgen05 stores waited
// for and fenced) before the warp's __syncwarp; the pair's MMA reads it only
// after rank 0 has seen the arrival.  A cluster-scope release per warp and
// stage measured 40 % slower on the emulated 8B-class GEMMs (and one
// relayed cluster-scope arrival per stage, 20 %).
__device__ __forceinline__ void mbar_arrive_rank0(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, 0;\n\t"
      "mbarrier.arrive.shared::cluster.b64 _, [ra];\n\t}" ::"r"(bar)
      : "memory");
}
// Parity probe that acquires at cluster scope (arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
static __device__ __noinline__ bool mbar_wait_cluster_slow(uint32_t bar, uint32_t parity,
                                                           volatile int* abort_flag, long long budget) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) return false;
  }
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  long long budget) {
  return mbar_try_wait_cluster(bar, parity) || mbar_wait_cluster_slow(bar, parity, abort_flag, budget);
}
// A device flag read once for the pair, before anything else the pair does:
// once both CTAs are known to run (a first cluster barrier, which is what
// makes the peer's shared memory addressable), thread 0 of rank 0 loads *flag
// and writes the value into the word at shared address `slot` in both CTAs;
// after a second barrier each thread reads its own CTA's copy.  Both CTAs
// therefore take the same branch even if the flag changes while the kernel
// runs, and either may return at once without touching the other's memory
// again.  Every thread of both CTAs calls it.
__device__ __forceinline__ int pair_read_flag(const int* flag, uint32_t slot) {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
  if (cluster_rank() == 0 && threadIdx.x == 0) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    asm volatile(
        "{\n\t.reg .b32 ra;\n\t"
        "st.shared.b32 [%0], %1;\n\t"
        "mapa.shared::cluster.u32 ra, %0, 1;\n\t"
        "st.shared::cluster.b32 [ra], %1;\n\t}" ::"r"(slot), "r"(v)
        : "memory");
  }
  cluster_sync();
  int v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(slot) : "memory");
  return v;
}
// TMEM of the pair: one warp of each CTA allocates (and later frees) the
// same columns in both CTAs' TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Arrive, once every MMA this thread issued before has completed, on the
// barrier at this offset in both CTAs of the pair.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((unsigned short)3)
      : "memory");
}

}  // namespace fp4q
