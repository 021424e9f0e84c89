// ws_sync.cuh -- synchronisation helpers of the warp-specialised tcgen05
// kernels: named-barrier votes, non-blocking and sleeping mbarrier waits,
// cp.async and per-warp mbarrier arrivals, ex2.
#pragma once

#include <stdint.h>

namespace csa {
namespace ws {

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ bool bar_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// Non-blocking: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Sleep on a barrier phase for at most about `ns` nanoseconds (returns either way).
__device__ __forceinline__ void mbar_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%0], %1, %2;\n}\n" ::"r"(bar), "r"(parity),
      "r"(ns)
      : "memory");
}
__device__ __forceinline__ void arrive_cp_async(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void arrive_warp(uint32_t bar) {  // 32 arrivals at once (lane 0)
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], 32;\n" ::"r"(bar) : "memory");
}


}  // namespace ws
}  // namespace csa
