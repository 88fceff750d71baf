// Inline-PTX helpers shared by the TMA / bulk-copy kernels: shared-memory addresses,
// mbarriers (init, expect-tx arrival, bounded parity wait) and bulk async copies.
#pragma once

#include <cstdint>

#include "ft_internal.cuh"

namespace ft {
namespace ptx {

constexpr uint32_t kWaitLimit = 1u << 24;  // try_wait polls before a wait gives up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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

// Bulk async copy global -> shared (16-byte aligned, size a multiple of 16), completing
// `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *counter >= target, for counters that other CTAs of the same grid
// raise (every CTA of that grid is resident: one CTA per SM, grid <= SM count).  Gives up
// after limit_ns (error word + abort flag) so that a lost signal cannot hang the GPU.
constexpr uint64_t kFlagWaitNs = 2000000000ull;  // 2 s
__device__ __forceinline__ bool wait_counter(const uint32_t* counter, uint32_t target, volatile int* abort_flag,
                                             uint32_t* error_word, uint64_t limit_ns = kFlagWaitNs) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (ld_acquire_gpu(counter) >= target) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) break;
    __nanosleep(64);
  }
  *abort_flag = 1;
  atomicOr(error_word, FT_DEVERR_TIMEOUT);
  return false;
}

// try_wait that lets the thread be suspended for up to `ns` while the phase is incomplete
// (it resumes as soon as the phase completes), instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of parity `parity`.  A waiting thread is suspended rather than
// polling, so warps that wait take no issue slots from the warps of the same SM that work.
// Gives up after kFlagWaitNs (error word + abort flag).
constexpr uint32_t kSuspendHintNs = 2000;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* error_word) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait_suspend(bar, parity, kSuspendHintNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kFlagWaitNs) break;
  }
  *abort_flag = 1;
  atomicOr(error_word, FT_DEVERR_TIMEOUT);
  return false;
}

// L2 policy for data read once per step (expert weights): evicted first, so that the
// small per-step state, activations and kernel code stay resident in L2 across kernels.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

}  // namespace ptx
}  // namespace ft
