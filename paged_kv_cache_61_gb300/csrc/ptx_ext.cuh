// sm_100-and-later device helpers of the MLA kernels: a non-blocking mbarrier test and a
// stall watchdog for the MMA-issuing polling loops, three-input min/max and paired f32
// arithmetic for the softmax rows.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace pda {
namespace ptx {

// Non-blocking test of the phase (try_wait may suspend the thread for a while when the
// phase is incomplete, which a thread polling several barriers in turn cannot afford).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Stall watchdog of a polling loop: it reads the global timer only while the loop makes no
// progress, once every 64 idle polls, so a loop that keeps issuing work pays nothing.
struct Watchdog {
  uint64_t t0 = 0;
  uint32_t idle = 0;
  __device__ __forceinline__ void progress() { idle = 0; }
  // An idle poll; true once the loop has made no progress for kWaitLimitNs.
  __device__ __forceinline__ bool expired() {
    const uint32_t n = idle++;
    if ((n & 63u) != 0) return false;
    const uint64_t now = globaltimer();
    if (n == 0) {
      t0 = now;
      return false;
    }
    return now - t0 > kWaitLimitNs;
  }
};

// Three-input maximum / minimum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pairs of f32 (one 64-bit register pair) and the paired FMA-pipe operations of
// sm_100 and later: half the issue slots of two scalar operations.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

}  // namespace ptx
}  // namespace pda
