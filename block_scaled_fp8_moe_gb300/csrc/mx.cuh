// Device helpers of the MX formats shared by the kernels: the round-up UE8M0 scale rule and
// E4M3 / E2M1 element encoders ("New Deepseek 4.1 flash recipe", post 6 "How it works" items 1-3).
#pragma once
#include <cstdint>

namespace moe {

// Smallest s with amax <= qmax * 2^s, where qmax = (1 + qm / 2^23) * 2^qe; exact integer work on
// the bits of amax, clamped to the UE8M0 range; amax = 0 -> -127.
__device__ __forceinline__ int mx_scale_exp(float amax, int qe, uint32_t qm) {
  uint32_t b = __float_as_uint(amax);
  if (b == 0) return -127;
  int e = (int)((b >> 23) & 0xFF);
  uint32_t man = b & 0x7FFFFF;
  if (e == 0) {                       // subnormal amax: normalise
    int sh = __clz(man) - 8;
    man = (man << sh) & 0x7FFFFF;
    e = 1 - sh;
  }
  int s = (e - 127) - qe + (man > qm ? 1 : 0);
  return max(-127, min(126, s));      // 127 is unreachable for finite fp32 amax and both formats
}
__device__ __forceinline__ int e4m3_scale_exp(float amax) { return mx_scale_exp(amax, 8, 0x600000u); }  // 448
__device__ __forceinline__ int e2m1_scale_exp(float amax) { return mx_scale_exp(amax, 2, 0x400000u); }  // 6

// 2^-s for s in [-127, 126] (always a normal fp32)
__device__ __forceinline__ float pow2_neg(int s) { return __uint_as_float((uint32_t)(127 - s) << 23); }

// Two E4M3 codes (round to nearest even, saturating -- never reached under the scale rule),
// `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// E2M1 round-to-nearest-even of v (|v| <= 6 under the scale rule), from the value grid
// {0, .5, 1, 1.5, 2, 3, 4, 6}: each comparison counts one grid step passed; at an exact midpoint
// the step is taken only when it lands on the even code.
__device__ __forceinline__ uint32_t e2m1_code(float v) {
  float a = fabsf(v);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return c | (signbit(v) ? 8u : 0u);
}

}  // namespace moe
