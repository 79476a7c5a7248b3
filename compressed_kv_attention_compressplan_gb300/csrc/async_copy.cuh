// async_copy.cuh -- mbarrier and bulk-copy (TMA engine) helpers shared by the
// kernels that stage data in shared memory (sm_90+ PTX, used on sm_103a).
//
// Every wait is bounded: it gives up after a time limit and reports it, so a
// copy that never completes turns into a status bit instead of a hung kernel.
// The ordinary waits of a kernel use the limit passed in its arguments
// (ckv_set_wait_limit_ns); a CTA that gives up still waits, with the fixed
// kWaitLimitNs, for the copies it has issued to land before it exits, so that
// no copy writes into shared memory the CTA no longer owns.
//
// try_wait may hold a thread until the phase completes when that happens
// within a hardware-chosen window of microseconds, so a limit shorter than
// that window can only be observed by polling test_wait.  Each staged kernel
// is therefore built twice: for limits of 1 ms and more (try_wait, the limit
// read only once a first probe has failed) and for shorter ones (test_wait
// polled against the timer); the launchers pick by the limit.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ckv {

// 2 s, far beyond any real copy: the default limit of the ordinary waits, and
// the limit of the waits for copies in flight before a CTA exits
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// the largest limit ckv_set_wait_limit_ns accepts (10 s); larger values are
// clamped to it, so every wait stays bounded
constexpr uint64_t kWaitLimitMaxNs = 10000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// The same test without suspending the thread (test_wait never blocks).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Limits below this (1 ms) are polled with test_wait, by kernels built for
// short waits (the kShortWaits instantiations, launched only for such limits).
constexpr uint64_t kShortWaitNs = 1000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase of parity `parity` to complete, for at most about
// `limit_ns` beyond try_wait's own window.  The first probe is the whole cost
// of a phase that completes on time; the limit is read only after it.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// The same with a limit below try_wait's window: test_wait polled against
// the timer.
__device__ __forceinline__ bool mbar_poll_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_test_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// A kernel's ordinary wait on one of its copies.
template <bool kShortWaits>
__device__ __forceinline__ bool wait_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return kShortWaits ? mbar_poll_bounded(bar, parity, limit_ns) : mbar_wait_bounded(bar, parity, limit_ns);
}

// The same wait by all 32 lanes of a warp, which then take one decision: the
// phase counts as complete only if every lane saw it complete.  After a
// timeout the whole warp therefore leaves together, and no lane is left
// waiting in a later warp-wide shuffle or __syncwarp for lanes that left.
template <bool kShortWaits>
__device__ __forceinline__ bool warp_wait_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xFFFFFFFFu, wait_for<kShortWaits>(bar, parity, limit_ns));
}

// An L2 prefetch of `bytes` (a multiple of 16) from the 16-byte aligned
// global address p.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// One bulk global -> shared copy that completes `bytes` of the barrier's
// transaction count.  dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

}  // namespace ckv
