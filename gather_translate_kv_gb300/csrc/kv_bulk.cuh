// Bulk copies between global and shared memory (the bulk-copy engine of
// sm_90+ GPUs, cp.async.bulk), with loads counted on an mbarrier and waits
// that give up after a bounded number of polls. Used by the fan-out gather
// (kv_gather.cu) and the bulk-copy move (kv_move.cu).
//
// A wait that runs out means a load never completed: the kernel ORs
// KV_DEV_ERR_TIMEOUT into the pool's error word, gives the loads in flight one
// more bounded wait, waits for its own bulk stores and returns, so the context
// stays usable. GTKV_TEST_EXTRA_TX makes every load barrier expect that many
// bytes more than its loads deliver; only the test build that checks this
// path sets it.
#pragma once

#include "kv_common.cuh"

#ifndef GTKV_TEST_EXTRA_TX
#define GTKV_TEST_EXTRA_TX 0
#endif

namespace gtkv {

constexpr uint32_t kBulkSpinLimit = 1u << 24;  // barrier polls before a load is given up on (~1 s)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One arrival per phase: the thread that issues a phase's loads.
__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive on the barrier and expect `bytes` from the loads of this phase.
__device__ __forceinline__ void mbar_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes + GTKV_TEST_EXTRA_TX)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Polls the barrier's phase `parity` at most kBulkSpinLimit times.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kBulkSpinLimit; ++i)
    if (mbar_test(bar, parity)) return true;
  return false;
}

// global -> shared, completion counted on `bar` (16-byte aligned addresses,
// bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// shared -> global, in the issuing thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// The issuing thread's bulk stores have read their shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// The issuing thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace gtkv
