// Top-k of one token's routing keys on one warp, shared by the router's plan kernels and the
// one-launch decode layer so that both make the same choices and compute the same weights.
// "New Deepseek 4.1 flash recipe": post 6 "How it works" item 3 (the MoE top-k gate); post 4
// "Exact indexer selections" (ties break by the lowest index).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

// One token's top-k on one warp. Lane l holds experts l, l + 32, ... (NI of them), sorted once in
// registers by (key desc, expert asc); each round is a warp arg-max over the lanes' heads (two warp
// reductions: the largest key, then the lowest expert holding it), after which the winning lane
// drops its head (a predicated shift, no divergent rescan). Selected weights: sigma_j / sum, the
// sum accumulated in rank order (identical on every lane). Lane j < k ends with the j-th choice.
// kPairs: krow holds (key, score) pairs, one 8-byte load per expert; srow is not read.
template <int NI, bool kPairs = false>
__device__ __forceinline__ void warp_topk(const float* __restrict__ krow, const float* __restrict__ srow, int E, int k,
                                          int lane, int16_t* sidx, int* my_e, float* my_s, float* sum_out) {
  // lane l holds experts e = l + 32 i: the key as an order-preserving unsigned image (keys are never
  // -0 or NaN, so every key maps above 0; 0 marks "nothing"), its score and its id
  uint32_t ku[NI];
  float sv[NI];
  int ev[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    const bool in = e < E;
    // through L2: another kernel wrote them
    float2 ks = make_float2(0.f, 0.f);
    if (kPairs && in) ks = __ldcg(reinterpret_cast<const float2*>(krow) + e);
    const uint32_t bits = in ? __float_as_uint(kPairs ? ks.x : __ldcg(krow + e)) : 0u;
    ku[i] = in ? ((bits & 0x80000000u) ? ~bits : (bits | 0x80000000u)) : 0u;
    sv[i] = in ? (kPairs ? ks.y : __ldcg(srow + e)) : 0.f;
    ev[i] = in ? e : 0x7fffffff;
  }
  // each lane sorts its items best first, (key desc, id asc), with a bitonic network in registers
#pragma unroll
  for (int size = 2; size <= NI; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool j_better = ku[j] > ku[i] || (ku[j] == ku[i] && ev[j] < ev[i]);
          const bool swap = ((i & size) == 0) ? j_better : !j_better;
          const uint32_t tk = ku[i];
          const float ts = sv[i];
          const int te = ev[i];
          ku[i] = swap ? ku[j] : ku[i];
          sv[i] = swap ? sv[j] : sv[i];
          ev[i] = swap ? ev[j] : ev[i];
          ku[j] = swap ? tk : ku[j];
          sv[j] = swap ? ts : sv[j];
          ev[j] = swap ? te : ev[j];
        }
      }
  // k rounds over the lanes' heads: the largest key, then the lowest id holding it; the winning
  // lane drops its head
  float sel_sum = 0.f;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, ku[0]);
    const int be = __reduce_min_sync(0xffffffffu, ku[0] == m ? ev[0] : 0x7fffffff);
    const float sc = __shfl_sync(0xffffffffu, sv[0], be & 31);
    const bool win = ev[0] == be;
#pragma unroll
    for (int i = 0; i + 1 < NI; ++i) {
      ku[i] = win ? ku[i + 1] : ku[i];
      sv[i] = win ? sv[i + 1] : sv[i];
      ev[i] = win ? ev[i + 1] : ev[i];
    }
    if (win) {
      ku[NI - 1] = 0u;
      ev[NI - 1] = 0x7fffffff;
    }
    sel_sum = __fadd_rn(sel_sum, sc);
    if (lane == j) { *my_e = be; *my_s = sc; }
    if (sidx && lane == 0) sidx[j] = (int16_t)be;
  }
  *sum_out = sel_sum;
}

}  // namespace moe
