// Asynchronous-copy pipeline helpers for sm_100-family GPUs: mbarriers,
// bulk (TMA engine) copies global -> shared, bounded waits.
//
// Every wait is bounded by a clock budget; on expiry the caller records
// kStatusTimeout in the device status word and unwinds, so no kernel of this
// library can spin forever.
#pragma once
#include <stdint.h>

namespace exl3 {

constexpr long long kWaitBudgetCycles = 1000000000LL;  // ~0.5 s at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Bounded wait that also gives up as soon as any CTA has recorded a timeout
// in the device status word (bit 4), so a stuck pipeline ends the whole grid
// quickly instead of every CTA spending its own budget.  The status word (a
// global load) is read only every kStatusPollCycles, so a wait that needs
// a few retries is not slowed by memory round trips.  A wait that runs out
// of budget sets bit 4 itself; either way a false return means "stop issuing
// work and unwind".
constexpr long long kStatusPollCycles = 20000;  // ~10 us
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity,
                                                   int32_t* status,
                                                   long long budget = kWaitBudgetCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  long long next_poll = t0 + kStatusPollCycles;
  while (!mbar_try_wait(bar, parity)) {
    const long long now = clock64();
    if (now >= next_poll) {
      if (*reinterpret_cast<volatile int32_t*>(status) & 4) return false;
      if (now - t0 > budget) {
        atomicOr(status, 4);
        return false;
      }
      next_poll = now + kStatusPollCycles;
    }
  }
  return true;
}

// Teardown wait: bounded by the clock budget only (it ignores the status
// word), for draining copies and tensor-core work this CTA issued before it
// releases shared memory or TMEM.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > budget) return false;
  return true;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace exl3
