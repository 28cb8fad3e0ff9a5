// MX quantisation kernels (HBM-bound, coalesced 16-byte accesses) and the weight packer.
//
// MXFP8 activations / MXFP4 weights: "New Deepseek 4.1 flash recipe", post 6 "How it works"
// items 1-3 (block-scaled MMA for MXFP8 and FP8 x FP4; TileKernels' quantisation casts).
// Scale rule: the power of two rounded up from amax / qmax, so no element saturates.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

// 8 bf16 elements per thread, 4 threads per 32-block.
__global__ void quant_mxfp8_kernel(const uint4* __restrict__ x, uint2* __restrict__ q, uint8_t* __restrict__ s,
                                   long long n_groups) {
  pdl_trigger();
  pdl_wait();
  // The loop bound is uniform across the warp (the shuffles below need every lane).
  const unsigned lane = threadIdx.x & 31;
  for (long long g0 = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); g0 < n_groups;
       g0 += (long long)gridDim.x * blockDim.x) {
    const long long g = g0 + lane;
    const bool valid = g < n_groups;
    uint4 v = valid ? __ldg(x + g) : make_uint4(0, 0, 0, 0);
    float f[8];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const int se = e4m3_scale_exp(m);
    const float sc = pow2_neg(se);
    uint32_t lo = e4m3x2(f[0] * sc, f[1] * sc) | (e4m3x2(f[2] * sc, f[3] * sc) << 16);
    uint32_t hi = e4m3x2(f[4] * sc, f[5] * sc) | (e4m3x2(f[6] * sc, f[7] * sc) << 16);
    if (valid) {
      q[g] = make_uint2(lo, hi);
      if ((g & 3) == 0) s[g >> 2] = (uint8_t)(se + 127);
    }
  }
}

// 8 fp32 elements per thread, 4 threads per 32-block.
__global__ void quant_mxfp4_kernel(const float4* __restrict__ w, uint32_t* __restrict__ q, uint8_t* __restrict__ s,
                                   long long n_groups) {
  const unsigned lane = threadIdx.x & 31;
  for (long long g0 = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); g0 < n_groups;
       g0 += (long long)gridDim.x * blockDim.x) {
    const long long g = g0 + lane;
    const bool valid = g < n_groups;
    float4 a = valid ? __ldg(w + 2 * g) : make_float4(0, 0, 0, 0);
    float4 b = valid ? __ldg(w + 2 * g + 1) : make_float4(0, 0, 0, 0);
    float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const int se = e2m1_scale_exp(m);
    const float sc = pow2_neg(se);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) packed |= e2m1_code(f[i] * sc) << (4 * i);
    if (valid) {
      q[g] = packed;
      if ((g & 3) == 0) s[g >> 2] = (uint8_t)(se + 127);
    }
  }
}

// Packed weight tiles: codes 128 rows x 64 bytes, scales one 512-byte block per tile.
// W13 (gate_up = true): tile (e, m, kc) row r -> canonical row (r < 64 ? 64m + r : I + 64m + r - 64).
// W2: tile (e, n, kc) row r -> canonical row 128n + r. `rows_per_e` = canonical rows per expert,
// `K` = row length in elements.
__device__ __forceinline__ int pack_src_row(bool gate_up, int mt, int r, int I) {
  return gate_up ? (r < 64 ? 64 * mt + r : I + 64 * mt + (r - 64)) : 128 * mt + r;
}

// `chunk_bytes` = bytes of one row's 128-element K-chunk: 64 for E2M1 codes, 128 for E4M3 codes.
__global__ void pack_codes_kernel(const uint8_t* __restrict__ q, uint8_t* __restrict__ qp, int E, int MT, int KC,
                                  int rows_per_e, int K, int I, bool gate_up, int chunk_bytes) {
  // one thread per 16 packed bytes
  const int parts = chunk_bytes / 16;
  const long long total = (long long)E * MT * KC * 128 * parts;
  const int row_bytes = K * chunk_bytes / kTileK;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    int part = (int)(i % parts);
    long long rr = i / parts;
    int r = (int)(rr % 128);
    long long tile = rr / 128;
    int kc = (int)(tile % KC);
    long long em = tile / KC;
    int mt = (int)(em % MT);
    int e = (int)(em / MT);
    int src_row = pack_src_row(gate_up, mt, r, I);
    int byte0 = kc * chunk_bytes + part * 16;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (byte0 < row_bytes)
      v = *reinterpret_cast<const uint4*>(q + ((long long)e * rows_per_e + src_row) * row_bytes + byte0);
    *reinterpret_cast<uint4*>(qp + tile * (128LL * chunk_bytes) + r * chunk_bytes + part * 16) = v;
  }
}

__global__ void pack_scales_kernel(const uint8_t* __restrict__ s, uint8_t* __restrict__ sp, int E, int MT, int KC,
                                   int rows_per_e, int K, int I, bool gate_up) {
  const long long total = (long long)E * MT * KC * 512;
  const int nb = K / 32;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    int o = (int)(i & 511);
    long long tile = i >> 9;
    int kc = (int)(tile % KC);
    long long em = tile / KC;
    int mt = (int)(em % MT);
    int e = (int)(em / MT);
    // byte o = (r % 32) * 16 + (r / 32) * 4 + b
    int b = o & 3, r = ((o >> 4) & 31) + 32 * ((o >> 2) & 3);
    int src_row = pack_src_row(gate_up, mt, r, I);
    int blk = kc * 4 + b;
    uint8_t v = 127;   // 2^0 for K-blocks past the end (their codes are zero)
    if (blk < nb) v = s[((long long)e * rows_per_e + src_row) * nb + blk];
    sp[i] = v;
  }
}

// The same quantisation, written straight into plan order: the codes and scales of token t go to
// plan rows row_of_slot[t k + j] (j < k; -1 = no row), and also to q / s in token order when those
// are given. Replaces quantise-then-gather for the wide-tile GEMM path.
__global__ void quant_mxfp8_plan_kernel(const uint4* __restrict__ x, uint2* __restrict__ q, uint8_t* __restrict__ s,
                                        const int32_t* __restrict__ row_of_slot, int k, int H, long long n_groups,
                                        uint2* __restrict__ qp, uint8_t* __restrict__ sp) {
  pdl_trigger();
  pdl_wait();
  const unsigned lane = threadIdx.x & 31;
  const int g_row = H / 8;                      // 8-element groups per row
  for (long long g0 = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); g0 < n_groups;
       g0 += (long long)gridDim.x * blockDim.x) {
    const long long g = g0 + lane;
    const bool valid = g < n_groups;
    uint4 v = valid ? __ldg(x + g) : make_uint4(0, 0, 0, 0);
    float f[8];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const int se = e4m3_scale_exp(m);
    const float sc = pow2_neg(se);
    const uint32_t lo = e4m3x2(f[0] * sc, f[1] * sc) | (e4m3x2(f[2] * sc, f[3] * sc) << 16);
    const uint32_t hi = e4m3x2(f[4] * sc, f[5] * sc) | (e4m3x2(f[6] * sc, f[7] * sc) << 16);
    if (valid) {
      const long long t = g / g_row;
      const int c = (int)(g - t * g_row);
      if (q) {
        q[g] = make_uint2(lo, hi);
        if ((g & 3) == 0) s[g >> 2] = (uint8_t)(se + 127);
      }
      for (int j = 0; j < k; ++j) {
        const int prow = __ldg(row_of_slot + t * k + j);
        if (prow < 0) continue;
        qp[(long long)prow * g_row + c] = make_uint2(lo, hi);
        if ((c & 3) == 0) sp[(long long)prow * (H / 32) + (c >> 2)] = (uint8_t)(se + 127);
      }
    }
  }
}

int launch_quant_mxfp8_plan(int rows, int cols, int k, const uint16_t* x, uint8_t* q, uint8_t* s,
                            const int32_t* row_of_slot, uint8_t* qp, uint8_t* sp, cudaStream_t st) {
  long long groups = (long long)rows * cols / 8;
  if (groups == 0) return MOE_OK;
  int threads = 256;
  long long need = (groups + threads - 1) / threads;
  int blocks = (int)std::min<long long>(need, (long long)num_sms() * 8);
  return launch_pdl(quant_mxfp8_plan_kernel, dim3(blocks), dim3(threads), 0, st, reinterpret_cast<const uint4*>(x),
                    reinterpret_cast<uint2*>(q), s, row_of_slot, k, cols, groups, reinterpret_cast<uint2*>(qp), sp);
}

int launch_quant_mxfp8(int rows, int cols, const uint16_t* x, uint8_t* q, uint8_t* s, cudaStream_t st) {
  long long groups = (long long)rows * cols / 8;
  if (groups == 0) return MOE_OK;
  int threads = 256;
  long long need = (groups + threads - 1) / threads;
  int blocks = (int)std::min<long long>(need, (long long)num_sms() * 8);
  return launch_pdl(quant_mxfp8_kernel, dim3(blocks), dim3(threads), 0, st, reinterpret_cast<const uint4*>(x),
                    reinterpret_cast<uint2*>(q), s, groups);
}

}  // namespace moe

using namespace moe;

extern "C" int moe_quant_mxfp8_plan(const moe_shape* sh, const uint16_t* x, const int32_t* row_of_slot,
                                    uint8_t* xq_plan, uint8_t* xs_plan, uint8_t* xq, uint8_t* xs, void* stream) {
  if (!sh) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(sh)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (sh->T == 0) return MOE_OK;
  if (!x || !row_of_slot || !xq_plan || !xs_plan || (!xq) != (!xs)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(xq_plan) & 7) ||
      (reinterpret_cast<uintptr_t>(xq) & 7) || (reinterpret_cast<uintptr_t>(row_of_slot) & 3))
    return MOE_ERR_INVALID_ARG;
  return launch_quant_mxfp8_plan(sh->T, sh->H, sh->k, x, xq, xs, row_of_slot, xq_plan, xs_plan,
                                 static_cast<cudaStream_t>(stream));
}

extern "C" int moe_quant_mxfp8(int32_t rows, int32_t cols, const uint16_t* x, uint8_t* q, uint8_t* s,
                               void* stream) {
  if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (cols % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !s) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(q) & 7)) return MOE_ERR_INVALID_ARG;
  return launch_quant_mxfp8(rows, cols, x, q, s, static_cast<cudaStream_t>(stream));
}

// Dead verification rows from survival estimates (post 2, "Speculative decoding": rows below 0.2
// skip the expert weight reads): dead[t] = p[t] < threshold in fp32 (NaN stays live).
__global__ void dead_from_survival_kernel(const float* __restrict__ p, float threshold, uint8_t* __restrict__ dead,
                                          int T) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) dead[t] = (p[t] < threshold) ? 1 : 0;
}

extern "C" int moe_dead_from_survival(int32_t T, const float* p_survive, float threshold, uint8_t* dead,
                                      void* stream) {
  if (T < 0 || !(threshold == threshold)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!p_survive || !dead || (reinterpret_cast<uintptr_t>(p_survive) & 3)) return MOE_ERR_INVALID_ARG;
  dead_from_survival_kernel<<<(T + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(p_survive, threshold,
                                                                                          dead, T);
  return launch_status();
}

extern "C" int moe_quant_mxfp4(int32_t rows, int32_t cols, const float* w, uint8_t* q, uint8_t* s, void* stream) {
  if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (cols % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!w || !q || !s) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) & 15) || (reinterpret_cast<uintptr_t>(q) & 3)) return MOE_ERR_INVALID_ARG;
  long long groups = (long long)rows * cols / 8;
  int threads = 256;
  long long need = (groups + threads - 1) / threads;
  int blocks = (int)std::min<long long>(need, (long long)num_sms() * 8);
  quant_mxfp4_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const float4*>(w), reinterpret_cast<uint32_t*>(q), s, groups);
  return launch_status();
}

static size_t packed_bytes(int E, int MT, int KC, size_t* scale_bytes) {
  size_t tiles = (size_t)E * MT * KC;
  if (scale_bytes) *scale_bytes = tiles * kTileScaleBytes;
  return tiles * kTileCodeBytes;
}

extern "C" size_t moe_packed_w13_bytes(const moe_shape* sh, size_t* scale_bytes) {
  if (!shape_ok(sh)) return 0;
  return packed_bytes(sh->E, sh->I / 64, sh->H / kTileK, scale_bytes);
}

extern "C" size_t moe_packed_w2_bytes(const moe_shape* sh, size_t* scale_bytes) {
  if (!shape_ok(sh)) return 0;
  return packed_bytes(sh->E, sh->H / 128, ceil_div(sh->I, kTileK), scale_bytes);
}

static int pack_common(const moe_shape* sh, const uint8_t* q, const uint8_t* s, uint8_t* qp, uint8_t* sp,
                       void* stream, bool gate_up, int chunk_bytes = 64) {
  if (!sh || !q || !s || !qp || !sp) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(sh)) return MOE_ERR_UNSUPPORTED_SHAPE;
  for (const void* p : {(const void*)q, (const void*)qp})
    if (reinterpret_cast<uintptr_t>(p) & 15) return MOE_ERR_INVALID_ARG;
  const int E = sh->E;
  const int MT = gate_up ? sh->I / 64 : sh->H / 128;
  const int K = gate_up ? sh->H : sh->I;
  const int KC = ceil_div(K, kTileK);
  const int rows_per_e = gate_up ? 2 * sh->I : sh->H;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int blocks = num_sms() * 8;
  pack_codes_kernel<<<blocks, 256, 0, st>>>(q, qp, E, MT, KC, rows_per_e, K, sh->I, gate_up, chunk_bytes);
  int rc = launch_status();
  if (rc) return rc;
  pack_scales_kernel<<<blocks, 256, 0, st>>>(s, sp, E, MT, KC, rows_per_e, K, sh->I, gate_up);
  return launch_status();
}

extern "C" int moe_pack_w13(const moe_shape* sh, const uint8_t* q, const uint8_t* s, uint8_t* qp, uint8_t* sp,
                            void* stream) {
  return pack_common(sh, q, s, qp, sp, stream, true);
}

extern "C" int moe_pack_w2(const moe_shape* sh, const uint8_t* q, const uint8_t* s, uint8_t* qp, uint8_t* sp,
                           void* stream) {
  return pack_common(sh, q, s, qp, sp, stream, false);
}

// ---------------------------------------------------------------------------------------------
// Shared expert weights: dense MXFP8 (E4M3 codes, one byte per element), packed like the routed
// experts' tiles with 128 bytes per row and K-chunk (16 KB of codes per tile).
// ---------------------------------------------------------------------------------------------
static bool shared_shape_ok(const moe_shape* sh) { return sh && shape_ok(sh) && sh->E == 1 && sh->k == 1; }

extern "C" size_t moe_packed_shared_w13_bytes(const moe_shape* sh, size_t* scale_bytes) {
  if (!shared_shape_ok(sh)) return 0;
  return 2 * packed_bytes(1, sh->I / 64, sh->H / kTileK, scale_bytes);
}

extern "C" size_t moe_packed_shared_w2_bytes(const moe_shape* sh, size_t* scale_bytes) {
  if (!shared_shape_ok(sh)) return 0;
  return 2 * packed_bytes(1, sh->H / 128, ceil_div(sh->I, kTileK), scale_bytes);
}

extern "C" int moe_pack_shared_w13(const moe_shape* sh, const uint8_t* q, const uint8_t* s, uint8_t* qp,
                                   uint8_t* sp, void* stream) {
  if (!sh) return MOE_ERR_INVALID_ARG;
  if (!shared_shape_ok(sh)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return pack_common(sh, q, s, qp, sp, stream, true, 128);
}

extern "C" int moe_pack_shared_w2(const moe_shape* sh, const uint8_t* q, const uint8_t* s, uint8_t* qp,
                                  uint8_t* sp, void* stream) {
  if (!sh) return MOE_ERR_INVALID_ARG;
  if (!shared_shape_ok(sh)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return pack_common(sh, q, s, qp, sp, stream, false, 128);
}
