// wd_pipeline.cuh - shared-memory streaming pipeline: bulk async copies from
// global memory into a ring of shared-memory stages, tracked by mbarriers.
//
// One producer thread per CTA issues cp.async.bulk copies of contiguous weight
// rows into stage s and arms the stage's "full" barrier with the byte count;
// consumer warps wait on "full", compute from shared memory and arrive on the
// stage's "empty" barrier, which the producer waits on before refilling it.
// The number of bytes in flight is set by the ring (tens of KiB per CTA), not
// by registers, which is what a bandwidth-bound GEMV needs on GB300.
//
// Every wait is bounded (about 2 s of SM clock cycles): a wait that runs out
// returns false, the caller raises bit 1 of the error flag and leaves, so a
// broken invariant can never hang the GPU.
#pragma once

#include <stdint.h>

namespace wd {

constexpr long long kWaitLimitCycles = 4000000000ll;  // ~2 s at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the other threads and to the async proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

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

// Wait for the phase of parity `parity` of barrier `bar` to complete.
// Returns false if it has not completed within kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitLimitCycles) return false;
  return true;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory to this CTA's shared memory, completing on barrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Bulk copy global -> shared without an L2 cache hint.
__device__ __forceinline__ void bulk_g2s_nohint(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bounded wait for a phase (as mbar_wait); returns 0 as a token to add to the
// shared-memory addresses of the data the phase guards (so that plain-asm
// reads of them cannot be scheduled above the wait); `ok` is false if the wait
// ran out.
__device__ __forceinline__ uint32_t mbar_wait_token(uint32_t bar, uint32_t parity, bool& ok) {
  ok = mbar_wait(bar, parity);
  uint32_t t;
  asm volatile("mov.u32 %0, 0;" : "=r"(t) : "r"(ok ? 1u : 0u) : "memory");
  return t;
}

// L2 policy for data read exactly once per launch (weight rows): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy for data many CTAs re-read (a shared weight row, activations).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Ask L2 to fetch the whole 16-byte chunks of [p, p + bytes) from HBM (no
// registers, no shared memory, nothing to wait for).  The partial chunks at
// either end are left out, so nothing outside the range is touched.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uintptr_t lo = (a + 15u) & ~static_cast<uintptr_t>(15u);
  const uintptr_t hi = (a + bytes) & ~static_cast<uintptr_t>(15u);
  if (hi > lo)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"((uint32_t)(hi - lo))
                 : "memory");
}

// Barrier among `count` threads (a multiple of 32) of the CTA, id 1..15.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint2 lds_u32x2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

}  // namespace wd
