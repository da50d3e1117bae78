// mbarrier, TMA and tcgen05 wrappers (inline PTX, sm_100+ / sm_103a).
//
// Every wait is bounded: after kWaitLimitNs of polling it reports failure,
// the caller sets RPA_STATUS_TIMEOUT, stops issuing work and leaves through
// its normal exit (freeing tensor memory), so a stuck pipeline never hangs
// the GPU.
#pragma once

#include <cuda.h>  // CUtensorMap

#include "common.cuh"

namespace rpa {

// Limit of every bounded wait.  A test build sets a short one (and can make
// one wait never complete) to exercise the timeout path.
#ifndef RPA_WAIT_LIMIT_NS
#define RPA_WAIT_LIMIT_NS 2000000000ull  // 2 s
#endif
constexpr unsigned long long kWaitLimitNs = RPA_WAIT_LIMIT_NS;
// Test builds only: when nonzero, the producers never signal that the query
// tile of a unit has landed, so the first wait on it runs out.
#ifndef RPA_TEST_STALL_QUERY
#define RPA_TEST_STALL_QUERY 0
#endif

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that may suspend the thread for up to `hint_ns` inside the
// instruction (it returns as soon as the phase completes), so a waiting warp
// does not take issue slots from the warps sharing its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Waits for the phase of parity `parity` to complete; false on timeout or
// when *abort (shared, set by another role that timed out) becomes nonzero.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// mbar_wait without suspending: polls the barrier with test_wait (checking
// the abort flag and the time limit every 64 polls).  For a lone thread
// whose waits are short and on the critical path (the MMA-issuing thread of
// the prefill), where waking from a suspended try_wait costs more than the
// polling takes from the warps sharing its scheduler.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_poll(uint32_t bar, uint32_t parity,
                                               volatile int* abort) {
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// mbar_wait for a whole warp (all 32 lanes call it): every lane returns from
// its own bounded wait, then the warp agrees on one outcome.  Lanes that saw
// the abort flag at different moments would otherwise leave their loop
// apart, and the warp's next collective (a .sync.aligned tensor-memory load,
// an ldmatrix / mma.sync, a __syncwarp) would wait for lanes that never come.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// Waits for the phase of parity `parity` without looking at the abort flag:
// an aborting CTA uses it to let the asynchronous copies and tensor-core
// products it issued finish before it frees their shared or tensor memory
// and exits.  Bounded by the same limit; false if it gave up.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// All threads of named barrier `id` (count threads) vote: true iff every
// one of them passes true.  Used where threads must leave a loop together
// (a thread that left alone would leave the others waiting at the next
// named barrier, which has no time limit).
__device__ __forceinline__ bool named_bar_all(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Plain bulk copy (no tensor map): 16-byte aligned addresses, size % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy ones (TMA writes, tensor-core reads) of the same memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier among `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Byte offset of 16-byte chunk c of row r in a tile written by a 128-byte
// swizzled TMA box (rows of 128 bytes, 1024-byte aligned tile base).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace rpa
