// Bulk-copy (TMA) and mbarrier primitives for sm_90+ (inline PTX), and the
// library's per-device status word.
//
// Every wait here is bounded: after `limit` unsuccessful polls (each poll may
// suspend the thread for a while in hardware) it gives up, records the
// timeout in the device status word (and in its host-visible copy) and
// returns false. A kernel that sees a failed wait raises its abort flag and
// winds down; the host reads the word with ar_device_status, or the copy with
// ar_plan_query and before every execution.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ar {

// Bits of the status word.
enum : unsigned int { kStatusTimeout = 1u };

// The library's sticky per-device status word (read by ar_device_status).
// Defined here: only one translation unit (fused_tma.cu) includes this file.
__device__ unsigned int g_ar_status_word;

// Host-visible copy of the status word: one word of page-locked, mapped host
// memory per device, which the host reads without synchronising. Null until
// the host has published it (the first executing call on the device).
__device__ unsigned int* g_ar_status_host;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make the barrier initialisations visible to the async (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive once and announce `bytes` of bulk-copy transactions to come.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete, at most `limit`
// polls; stop early if *abort becomes non-zero. Returns false on timeout or
// abort (and records a timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit,
                                          volatile int* abort) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  atomicOr(&g_ar_status_word, kStatusTimeout);
  if (unsigned int* h = g_ar_status_host) {
    // Only one bit exists, so a plain store of it loses nothing to racing
    // writers; the fence makes it visible to the host before the kernel ends.
    *reinterpret_cast<volatile unsigned int*>(h) = kStatusTimeout;
    __threadfence_system();
  }
  *abort = 1;
  return false;
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned); completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared -> global bulk copy, tracked in the issuing thread's bulk group.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed store groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's committed store groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's ordinary shared-memory writes before later bulk copies
// that read them.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier among `threads` threads (a multiple of 32) of the CTA, on barrier id.
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace ar
