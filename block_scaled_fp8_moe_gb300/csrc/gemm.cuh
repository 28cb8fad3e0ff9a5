// Pieces shared by the grouped GEMM kernels (gemm.cu: one CTA per accumulator; gemm2sm.cu: CTA
// pairs issuing tcgen05 MMAs across two SMs): the kernel parameters, bounded-wait and plan-table
// helpers, the epilogue arithmetic, and the host-side tensor maps of the packed weights and the
// activation rows.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // one second

struct GemmParams {
  // B side (activations)
  const uint8_t* bq;        // W13: xq [T, H];  W2: hq [S, I]
  const uint8_t* bs;        // W13: xs [T, H/32]; W2: hs [S, HS_PITCH]
  int b_plan_rows;          // W13: 1 if bq/bs rows are plan rows (row p feeds plan row p), 0 if token rows
  int b_row_bytes;          // K in bytes (= elements)
  int b_scale_pitch;        // bytes per scale row
  // A side (packed weights)
  const uint8_t* a_codes;   // packed tiles (the tensor map's memory), for L2 prefetch
  const uint8_t* a_scales;  // packed 512-byte scale blocks
  int a_fp8;                // 0: E2M1 codes (8 KB packed tiles, unpacked by the TMA); 1: E4M3 (16 KB tiles)
  // plan
  const int32_t* offsets;   // [E + 1]
  const int32_t* slot_of_row;
  int E, k, K, KC, MT;      // MT = weight panels (of 128 packed rows) per expert
  int I, H;
  // W13 outputs
  uint8_t* hq;
  uint8_t* hs;
  int hs_pitch;
  float* dbg;
  // W2 output: per-slot rows in plan order, before the routing weight
  float* y;
  uint32_t* status;
  // W13 then W2 in one launch: W13 epilogue warps count finished tiles per expert in ready[0..E)
  // (after their stores), and a W2 tile gathers its expert's rows only once every W13 tile of that
  // expert has been counted; W2 epilogue warps count their finished tiles in ready[E]. Zeroed before
  // each layer call by the kernel that ran before this one (the plan kernel, or the decode router
  // when the GEMM plans for itself).
  uint32_t* ready;
  // ... and, when out is set, the fixed-order combine of the T rows at the end of the launch, once
  // ready[E] says every W2 tile is stored
  const float* topk_w;
  const int32_t* row_of_slot;
  uint16_t* out;
  int T;
  // One-launch decode layer (small batches): every CTA selects the top-k of the T rows from the
  // router's (key, score) pairs (CTA b reads copy b mod kSelfPlanReplicas of [T, E]) and builds
  // the plan in its own shared memory (rows the dead mask flags get no plan rows); CTA 0 also
  // writes the plan to the plan_* arrays for the caller.
  const float2* sel;
  const uint8_t* dead;
  int32_t* plan_topk_idx;
  float* plan_topk_w;
  int32_t* plan_counts;
  int32_t* plan_offsets;
  int32_t* plan_slot_of_row;
  int32_t* plan_row_of_slot;
};


// One lane waits (bounded), the whole warp learns the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort, uint32_t* err,
                                          uint32_t code) {
  uint32_t ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, kWaitLimitNs, abort, err, code) ? 1u : 0u;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The token operand's scale bytes of one 128-deep K-chunk, in the MMA's scale layout: per 128 tile
// rows one 512-byte atom whose 16-byte line j holds the 4 bytes (the chunk's four 32-blocks) of
// rows j, j + 32, j + 64 and j + 96. Lane j of the producer warp loads the words of its NA lines
// with plain loads (a row past nrows reads as zero, scale 2^-127, and is never stored by the
// epilogue) and later stores each line with one 16-byte shared store: 4 conflict-free wavefronts
// per atom, where 4-byte cp.async copies into the same layout cost one wavefront per lane.
template <int NA>
struct ScaleLines {
  uint32_t w[NA][4];
};

template <int NA>
__device__ __forceinline__ void load_scale_lines(ScaleLines<NA>& s, const uint8_t* bs, size_t pitch, int row0,
                                                 int nrows, int kc, int lane) {
#pragma unroll
  for (int a = 0; a < NA; ++a)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = 128 * a + 32 * q + lane;
      s.w[a][q] = c < nrows ? *reinterpret_cast<const uint32_t*>(bs + (size_t)(row0 + c) * pitch + kc * 4) : 0u;
    }
}

template <int NA>
__device__ __forceinline__ void store_scale_lines(const ScaleLines<NA>& s, uint8_t* atoms, int lane) {
#pragma unroll
  for (int a = 0; a < NA; ++a)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(atoms + a * 512 + lane * 16)),
                 "r"(s.w[a][0]), "r"(s.w[a][1]), "r"(s.w[a][2]), "r"(s.w[a][3])
                 : "memory");
}

__device__ __forceinline__ int find_expert(const int* cum, int E, int w) {
  // largest e with cum[e] <= w (cum non-decreasing, cum[E] > w)
  int lo = 0, hi = E;           // invariant: cum[lo] <= w < cum[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (cum[mid] <= w) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Bounded wait (one thread) until a counter in global memory reaches `need` (acquire: the writes
// published before each increment are visible afterwards). On expiry it records DEV_TIMEOUT_FULL
// in *err, sets *abort and returns false; it returns false at once if *abort is already set.
__device__ __forceinline__ bool wait_count_at_least(const uint32_t* counter, uint32_t need, uint64_t limit_ns,
                                                    volatile uint32_t* abort, uint32_t* err) {
  auto load = [&]() {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    return v;
  };
  if (load() >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (load() >= need) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      atomicCAS(err, 0u, (uint32_t)DEV_TIMEOUT_FULL);
      return false;
    }
    __nanosleep(64);
  }
}

// ---------------------------------------------------------------------------------------------
// Epilogue pieces, shared by the one-CTA and the CTA-pair grouped GEMMs so that every tile kind
// does the same arithmetic on an accumulator column.
// ---------------------------------------------------------------------------------------------

// W13: one 16-column chunk of a 128-row accumulator of weight panel m (TMEM lanes 0..63 gate
// features 64m.., lanes 64..127 the matching up features), read by the four warps q = 0..3 of one
// epilogue set (128 threads, thread t = 0..127 of the set, named barrier bar_id) into registers r.
// q 0,1 hold gate features 64m + 32q + lane, q 2,3 the matching up features. The chunk goes to
// shared memory as [column][feature]; then thread t owns column t / 8 and the eight features
// 8 (t % 8) .. +7: SwiGLU, a four-thread amax per 32-block, and one 8-byte store of codes.
// Feature f of a column sits at f ^ (4 * (f / 32 % 2)): the second 32-feature half has its float4
// slots swapped in pairs, so the eight 16-byte reads of a quarter-warp (features 8 j and 8 j + 4 of
// one column) fall on distinct banks. Every thread of the set calls this (ok = false after an
// expired wait, store = false for a panel past the expert's last one) so that all meet at the
// barriers.
__device__ __forceinline__ void epi_w13_chunk(const uint32_t (&r)[16], float* xchg_set, int q, int lane, int t,
                                              uint32_t bar_id, bool ok, bool store, int c0, int m, int row0,
                                              int nrows, const GemmParams& p) {
  float* gs = xchg_set;           // [16][64] gate
  float* us = gs + 16 * 64;       // [16][64] up
  if (ok) {
    float* dst = (q < 2) ? gs : us;
    const int fsw = (32 * (q & 1) + lane) ^ (4 * (q & 1));
#pragma unroll
    for (int c = 0; c < 16; ++c) dst[c * 64 + fsw] = __uint_as_float(r[c]);
  }
  named_bar_sync(bar_id, 128);
  if (ok) {
    const int cc = t >> 3, f0 = (t & 7) * 8;
    const int col = c0 + cc;
    const int s0 = f0 ^ (4 * (f0 >> 5)), s1 = (f0 + 4) ^ (4 * (f0 >> 5));
    const float4 g0 = *reinterpret_cast<const float4*>(gs + cc * 64 + s0);
    const float4 g1 = *reinterpret_cast<const float4*>(gs + cc * 64 + s1);
    const float4 u0 = *reinterpret_cast<const float4*>(us + cc * 64 + s0);
    const float4 u1 = *reinterpret_cast<const float4*>(us + cc * 64 + s1);
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float a[8];
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a[i] = silu_mul(gv[i], uv[i]);
      am = fmaxf(am, fabsf(a[i]));
    }
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    const int se = e4m3_scale_exp(am);
    const float sc = __uint_as_float((uint32_t)(127 - se) << 23);
    const uint32_t lo = e4m3x2(a[0] * sc, a[1] * sc) | (e4m3x2(a[2] * sc, a[3] * sc) << 16);
    const uint32_t hi = e4m3x2(a[4] * sc, a[5] * sc) | (e4m3x2(a[6] * sc, a[7] * sc) << 16);
    if (store && col < nrows) {
      const size_t prow = (size_t)(row0 + col);
      const int feat = 64 * m + f0;
      *reinterpret_cast<uint2*>(p.hq + prow * p.I + feat) = make_uint2(lo, hi);
      if ((t & 3) == 0) p.hs[prow * p.hs_pitch + (feat >> 5)] = (uint8_t)(se + 127);
      if (p.dbg) {
        float4* d = reinterpret_cast<float4*>(p.dbg + prow * p.I + feat);
        d[0] = make_float4(a[0], a[1], a[2], a[3]);
        d[1] = make_float4(a[4], a[5], a[6], a[7]);
      }
    }
  }
  named_bar_sync(bar_id, 128);
}

// W2: one 16-column chunk of a 128-row accumulator of output panel m, held by warp q (TMEM lanes
// 32q..32q+31): plan row row0 + c0 + c of the per-slot buffer gets features 128 m + 32 q + lane;
// each store instruction writes 128 contiguous bytes (the routing weight is applied by the combine).
// kStream: evict-first stores, for per-slot buffers that the combine reads only after the launch
// (prefill: gigabytes that no later step of the GEMM reads from L2); the one-launch decode kernel
// reads its rows back from L2 and stores them normally.
template <bool kStream>
__device__ __forceinline__ void epi_w2_chunk(const uint32_t (&r)[16], int q, int lane, int c0, int m, int row0,
                                             int nrows, const GemmParams& p) {
  const int feat = 128 * m + 32 * q + lane;
  float* yrow = p.y + (size_t)(row0 + c0) * p.H + feat;
#pragma unroll
  for (int c = 0; c < 16; ++c)
    if (c0 + c < nrows) {
      if (kStream) __stcs(yrow + (size_t)c * p.H, __uint_as_float(r[c]));
      else yrow[(size_t)c * p.H] = __uint_as_float(r[c]);
    }
}

// ---------------------------------------------------------------------------------------------
// Host side: tensor maps
// ---------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Packed weight codes viewed as [tiles * 128 rows, 128 FP4 elements], 64 bytes per row; one box
// covers `box_tiles` consecutive tiles.
inline int make_weight_tmap(CUtensorMap* m, const uint8_t* codes, long long tiles, int box_tiles) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  cuuint64_t gdim[2] = {128, (cuuint64_t)tiles * 128};
  cuuint64_t gstride[1] = {64};
  cuuint32_t box[2] = {128, (cuuint32_t)(128 * box_tiles)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t*>(codes), gdim, gstride, box,
                   estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Packed E4M3 weight codes viewed as [tiles * 128 rows, 128 bytes]; one box covers `box_tiles`
// consecutive tiles (the same 128-byte swizzled shared layout as the unpacked FP4 tiles).
inline int make_weight_tmap_fp8(CUtensorMap* m, const uint8_t* codes, long long tiles, int box_tiles) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  cuuint64_t gdim[2] = {128, (cuuint64_t)tiles * 128};
  cuuint64_t gstride[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)(128 * box_tiles)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Activation codes viewed as [rows, row_bytes] bytes, 128-byte swizzled boxes of box_rows rows.
inline int make_act_tmap(CUtensorMap* m, const uint8_t* base, int row_bytes, long long rows, int box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  cuuint64_t gdim[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// CTA-pair grouped GEMM (gemm2sm.cu) for wide token tiles: same inputs and results as the one-CTA
// kernel's wide tiles.
int launch_gemm_pair(const moe_shape* s, const uint8_t* codes, const GemmParams& gp, bool w13, cudaStream_t st);
// Weight-stationary down projection (gemm_ws.cu) for a short K with wide token tiles: same inputs
// and results as the one-CTA kernel's W2.
bool ws_down_supported(const moe_shape* s);
int launch_gemm_ws(const moe_shape* s, const uint8_t* codes, const GemmParams& gp, cudaStream_t st);

}  // namespace moe
