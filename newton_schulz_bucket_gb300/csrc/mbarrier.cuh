// mbarrier helpers with bounded waits (shared by the tcgen05 GEMM and the
// wait test hook).  No wait in this library spins forever: after a cycle
// budget the waiter raises an abort flag its CTA's other roles poll, sets a
// bit in the plan's device error word (read by muon_plan_check_error) and
// returns, so the kernel ends and the context stays usable.
#pragma once

#include <cstdint>

namespace muon {

constexpr long long kWaitCycles = 1ll << 32;  // ~2 s at 2 GHz

__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if another role aborted or the wait ran out (then the
// error word gets bit `code` and every role is told to stop).
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, volatile int* abort_flag,
                                          int* err, int code, long long limit = kWaitCycles) {
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      if (err) atomicOr(err, code);
      return false;
    }
  }
  return true;
}

}  // namespace muon
