// The fixed-order weighted combine of one token's routed slots, for eight consecutive hidden
// features: shared by the combine kernel and the tail of the one-launch decode GEMM, so both produce
// the same bits. TP4 serving profile README, settings table "Experts" row: a per-slot buffer and a
// fixed-order sum instead of atomics.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace moe {

// out[t, 8 h8 .. 8 h8 + 7] = bf16_rne( ((w_0 y[r_0] + w_1 y[r_1]) + ...) + w_{k-1} y[r_{k-1}]
// (+ y_shared[t]) ), r_j = row_of_slot[t k + j], w_j = topk_w[t k + j]; each w_j y is one fp32
// multiply, the sum a left fold in fp32. Rows without slots (row_of_slot[t k] < 0) and rows the dead
// mask flags get +0.0; a flagged row that still holds slots is recorded in *status.
// kL2Only: y was written earlier in the same launch by other SMs, so it is read through L2 only;
// otherwise (the combine kernel) each y row is read exactly once, with evict-first loads.
// kPlanShared: topk_w and row_of_slot point to shared memory (plain loads, not the read-only path).
template <bool kL2Only, bool kPlanShared = false>
__device__ __forceinline__ void combine_unit(const float* __restrict__ y, const float* __restrict__ topk_w,
                                             const int32_t* __restrict__ row_of_slot, int t, int h8, int H, int k,
                                             uint16_t* __restrict__ out, const float* __restrict__ y_shared,
                                             const uint8_t* __restrict__ dead, uint32_t* status) {
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  const bool held = row_of_slot[(size_t)t * k] >= 0;
  const bool flagged = dead != nullptr && dead[t] != 0;
  if (flagged && held && h8 == 0 && status) atomicCAS(status, 0u, (uint32_t)DEV_BAD_INPUT);
  if (held && !flagged) {
    for (int j = 0; j < k; ++j) {
      const int r = kPlanShared ? row_of_slot[(size_t)t * k + j] : __ldg(row_of_slot + (size_t)t * k + j);
      const float w = kPlanShared ? topk_w[(size_t)t * k + j] : __ldg(topk_w + (size_t)t * k + j);
      const float4* yp = reinterpret_cast<const float4*>(y + (size_t)r * H) + 2 * h8;
      const float4 a = kL2Only ? __ldcg(yp) : __ldcs(yp);
      const float4 b = kL2Only ? __ldcg(yp + 1) : __ldcs(yp + 1);
      const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float wv = __fmul_rn(w, v[q]);
        acc[q] = (j == 0) ? wv : __fadd_rn(acc[q], wv);
      }
    }
    if (y_shared) {
      const float4* yp = reinterpret_cast<const float4*>(y_shared + (size_t)t * H) + 2 * h8;
      const float4 a = __ldg(yp), b = __ldg(yp + 1);
      const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], v[q]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q] + 0.0f));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q + 1] + 0.0f));
    o[q] = lo | (hi << 16);
  }
  *reinterpret_cast<uint4*>(out + (size_t)t * H + 8 * h8) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace moe
