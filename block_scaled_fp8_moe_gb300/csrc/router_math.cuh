// Router arithmetic shared by the router kernels: a library-independent fp32 exp/sigmoid and
// bf16 unpacking ("New Deepseek 4.1 flash recipe", post 6 "How it works" item 3: the MoE top-k
// gate; post 6 "Why TileLang": fixed-order reductions).
#pragma once
#include <cstdint>

namespace moe {

// ---------------------------------------------------------------------------------------------
// Library-independent exp / sigmoid from IEEE fp32 +, -, *, / (each correctly rounded; the
// _rn intrinsics keep the compiler from contracting them). exp(t), t in [-80, 80]:
// n = rint(t / ln2); r = (t - n ln2_hi) - n ln2_lo (Cody & Waite); degree-7 Taylor polynomial
// of exp(r) in Horner form; times 2^n (exact). ln2_hi keeps 16 significant bits so n * ln2_hi
// is exact. Coefficients are 1/k! rounded to fp32.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float exp_cw(float t) {
  const float kLog2e = 1.4426950408889634f;
  const float kLn2Hi = 0.693145751953125f;              // 45426 / 2^16
  const float kLn2Lo = 1.4286067653302226e-06f;         // ln2 - kLn2Hi, rounded to fp32
  float n = rintf(__fmul_rn(t, kLog2e));
  float r = __fsub_rn(t, __fmul_rn(n, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
  float p = 1.9841269841269841e-04f;                    // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), 1.3888888888888889e-03f);   // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), 8.3333333333333332e-03f);   // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), 4.1666666666666664e-02f);   // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), 1.6666666666666666e-01f);   // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const float two_n = __int_as_float(((int)n + 127) << 23);
  return __fmul_rn(p, two_n);
}

__device__ __forceinline__ float sigmoid_cw(float z) {
  float t = fminf(fmaxf(-z, -80.0f), 80.0f);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_cw(t)));
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// acc <- fma(lo(x), lo(w), acc), then the same for the high halves (elements 2i, 2i + 1): fp32
// fused multiply-add of bf16 operands, one rounding per step -- the same value as widening first.
__device__ __forceinline__ float fma2_bf16(uint32_t x, uint32_t w, float acc) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
      "mov.b32 {xl, xh}, %1;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
      "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}"
      : "+f"(acc)
      : "r"(x), "r"(w));
  return acc;
}

}  // namespace moe
