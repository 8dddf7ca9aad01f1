// Device helpers shared by the decode kernels: the approximate exp2 used for
// softmax numerators, a drain wait for in-flight copies, and the transposed
// warp butterflies that reduce per-lane head vectors over the lanes of a warp
// (64 heads over 32 lanes) or of a half-warp (32 heads over 16 lanes).
#pragma once

#include "ptx.cuh"

namespace skv {

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (the three-input form of max.f32, sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The max of 32 values: 17 operations, four deep (a chain of two-input maxima
// takes 31).
__device__ __forceinline__ float max32(const float (&x)[32]) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = fmax3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  a[10] = fmaxf(x[30], x[31]);
  const float b0 = fmax3(a[0], a[1], a[2]), b1 = fmax3(a[3], a[4], a[5]), b2 = fmax3(a[6], a[7], a[8]);
  return fmaxf(fmax3(b0, b1, b2), fmaxf(a[9], a[10]));
}

// Waits without looking at the abort flag (used to drain in-flight copies on abort).
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Transposed butterfly over a warp: each lane holds x[j] for 64 heads j; on
// return lane l holds the reduction over all 32 lanes for heads 2l and 2l+1.
template <bool kMax>
__device__ __forceinline__ void warp_transpose_reduce(const float (&x)[64], int lane, float& r0,
                                                      float& r1) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a[32];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float send = up ? x[i] : x[i + 32];
      const float keep = up ? x[i + 32] : x[i];
      a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
  }
  float b[16];
  {
    const bool up = lane & 8;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float send = up ? a[i] : a[i + 16];
      const float keep = up ? a[i + 16] : a[i];
      b[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
  }
  float c[8];
  {
    const bool up = lane & 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float send = up ? b[i] : b[i + 8];
      const float keep = up ? b[i + 8] : b[i];
      c[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
  }
  float d[4];
  {
    const bool up = lane & 2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = up ? c[i] : c[i + 4];
      const float keep = up ? c[i + 4] : c[i];
      d[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
  }
  {
    const bool up = lane & 1;
    const float send0 = up ? d[0] : d[2];
    const float keep0 = up ? d[2] : d[0];
    const float send1 = up ? d[1] : d[3];
    const float keep1 = up ? d[3] : d[1];
    r0 = op(keep0, __shfl_xor_sync(0xffffffffu, send0, 1));
    r1 = op(keep1, __shfl_xor_sync(0xffffffffu, send1, 1));
  }
}


// The same over each half of a warp: each lane holds x[j] for 32 heads j; on
// return lane l holds the reduction over the 16 lanes of its half-warp for heads
// 2(l mod 16) and 2(l mod 16)+1. The two halves never exchange values.
template <bool kMax>
__device__ __forceinline__ void halfwarp_transpose_reduce(const float (&x)[32], int lane, float& r0,
                                                          float& r1) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float b[16];
  {
    const bool up = lane & 8;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float send = up ? x[i] : x[i + 16];
      const float keep = up ? x[i + 16] : x[i];
      b[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
  }
  float c[8];
  {
    const bool up = lane & 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float send = up ? b[i] : b[i + 8];
      const float keep = up ? b[i + 8] : b[i];
      c[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
  }
  float d[4];
  {
    const bool up = lane & 2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = up ? c[i] : c[i + 4];
      const float keep = up ? c[i + 4] : c[i];
      d[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
  }
  {
    const bool up = lane & 1;
    const float send0 = up ? d[0] : d[2];
    const float keep0 = up ? d[2] : d[0];
    const float send1 = up ? d[1] : d[3];
    const float keep1 = up ? d[3] : d[1];
    r0 = op(keep0, __shfl_xor_sync(0xffffffffu, send0, 1));
    r1 = op(keep1, __shfl_xor_sync(0xffffffffu, send1, 1));
  }
}

}  // namespace skv
