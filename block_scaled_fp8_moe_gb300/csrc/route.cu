// Router (fixed-order fp32 logits, self-written sigmoid, top-k with lowest-index ties), expert
// plan (deterministic counting sort), and the fixed-order combine.
//
// "New Deepseek 4.1 flash recipe": post 6 "How it works" item 3 (TileKernels MoE top-k gate);
// post 6 "Why TileLang" (every reduction in a fixed order, batch-invariant rows); post 4
// "Exact indexer selections" (ties break by lowest position); post 2 (dead verification rows).
// TP4 serving profile README, "Experts" row: per-slot buffer + fixed-order sum instead of atomics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "combine.cuh"
#include "common.cuh"
#include "mx.cuh"
#include "ptx.cuh"
#include "router_math.cuh"
#include "topk.cuh"

namespace moe {

// ---------------------------------------------------------------------------------------------
// Logits, small T (decode): one warp per expert. Lane l owns the chunks c = l, l + 32, ...;
// each chunk is a sequential fma chain from +0; chunk sums go to shared memory and lane t folds
// them left to right for token t.
// ---------------------------------------------------------------------------------------------
constexpr int kSmallT = 16;

__global__ void __launch_bounds__(256) router_small_kernel(const uint16_t* __restrict__ x,
                                                           const uint16_t* __restrict__ wr,
                                                           const float* __restrict__ bias, int T, int H, int E,
                                                           float* __restrict__ score, float* __restrict__ key) {
  pdl_trigger();
  pdl_wait();
  __shared__ float part[8][kSmallT][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  if (e >= E) return;
  const int NC = H / kRouterChunk;
  float acc = 0.f;                                     // lane t < T folds token t
  for (int c0 = 0; c0 < NC; c0 += 32) {
    const int c = c0 + lane;
    if (c < NC) {
      const uint4* wp = reinterpret_cast<const uint4*>(wr + (size_t)e * H + (size_t)c * kRouterChunk);
      uint4 wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) wv[i] = __ldg(wp + i);
      for (int t = 0; t < T; ++t) {
        const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)t * H + (size_t)c * kRouterChunk);
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 xv = __ldg(xp + i);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            p = __fmaf_rn(bf_lo(xw[q]), bf_lo(ww[q]), p);
            p = __fmaf_rn(bf_hi(xw[q]), bf_hi(ww[q]), p);
          }
        }
        part[warp][t][lane] = p;
      }
    }
    __syncwarp();
    if (lane < T) {
      const int n = min(32, NC - c0);
      for (int i = 0; i < n; ++i) acc = __fadd_rn(acc, part[warp][lane][i]);
    }
    __syncwarp();
  }
  if (lane < T) {
    const float sc = sigmoid_cw(acc);
    score[(size_t)lane * E + e] = sc;
    key[(size_t)lane * E + e] = __fadd_rn(sc, bias[e]);
  }
}

// ---------------------------------------------------------------------------------------------
// Logits, small T (decode). The grid is (expert blocks of epc experts) x (token blocks of up to tpc
// rows). A CTA stages its token block's rows of x in shared memory by cp.async (every 16-byte copy
// in flight at once; chunk pitch 144 B so a quarter-warp's 16-byte reads of consecutive chunks hit
// distinct banks). Thread (g, c) owns chunk c of the EPT experts g EPT .. g EPT + EPT - 1 of the
// block: it loads their 128-byte Wr chunks into registers once and, for every staged token, runs
// the sequential fma chain of the chunk for each of them (bf16 operands, fp32 accumulate; two
// tokens at a time, as independent chains). The chunk partials go to shared memory, then one
// thread per (expert, token) folds them left to right and applies the sigmoid: the same order as
// router_small_kernel and the tiled kernel. Optionally the CTAs of a token block also
// MXFP8-quantise its rows, each a share of the 32-blocks.
// ---------------------------------------------------------------------------------------------
constexpr int kDecMaxT = 64;
constexpr int kDecThreadsMax = 512;
constexpr size_t kDecodeSmemMax = 210 * 1024;
constexpr int kDecPitch = 144;      // bytes per staged 64-element chunk
constexpr int kDecSmallT = 16;      // up to this many rows: kDecEpcSmall experts per CTA,
constexpr int kDecEpcSmall = 2;
constexpr int kDecTpcSmall = 2;     // ... blocks of this many rows
constexpr int kDecEpcLarge = 8;     // more rows: blocks of kDecTpcLarge rows, kDecEpcLarge experts per CTA
constexpr int kDecTpcLarge = 8;

struct DecodeRouterCfg {
  int ept, epc, tpc, threads;
  size_t smem;
};

// Up to kDecSmallT rows: blocks of two rows and two experts per CTA (one per thread; the Wr stream
// is spread over E / 2 CTAs per block). Every CTA staging all the rows had each L2 line of x read
// by all E / 2 CTAs at once: two-row blocks were the fastest of 1, 2, 3 and all 6 at decode-6.
// Beyond that: blocks of 8 rows and eight experts per CTA (two per thread), so that each CTA
// stages few rows of x and serves many experts with them (16-row blocks: the same at 48 rows,
// 4 us slower at 32).
inline DecodeRouterCfg decode_router_cfg(int T, int H, int E) {
  const int NC = H / kRouterChunk;
  DecodeRouterCfg c{};
  const bool small = T <= kDecSmallT;
  c.ept = small ? 1 : 2;
  c.epc = small ? kDecEpcSmall : kDecEpcLarge;
  if (c.epc > E) c.epc = E;
  c.tpc = small ? std::min(T, kDecTpcSmall) : kDecTpcLarge;
  c.threads = ((c.epc + c.ept - 1) / c.ept) * NC;
  auto smem = [&](int tpc) { return (size_t)tpc * NC * kDecPitch + (size_t)c.epc * tpc * (NC + 1) * 4; };
  while (c.tpc > 1 && smem(c.tpc) > kDecodeSmemMax) --c.tpc;
  c.smem = smem(c.tpc);
  return c;
}

template <int EPT>
__global__ void __launch_bounds__(kDecThreadsMax) router_decode_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, const float* __restrict__ bias, int T, int H,
    int E, int epc, int tpc, float* __restrict__ score, float* __restrict__ key, uint8_t* __restrict__ xq,
    uint8_t* __restrict__ xs, uint32_t* __restrict__ ready, float2* __restrict__ sel) {
  pdl_trigger();
  pdl_wait();
  // the one-launch W13 + W2 GEMM's counters (nullable), when no plan kernel runs in between
  if (ready && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i <= E; i += blockDim.x) ready[i] = 0;
  extern __shared__ __align__(16) uint8_t dsm_dec[];
  const int NC = H / kRouterChunk;
  const int t0 = blockIdx.y * tpc;
  const int tn = min(tpc, T - t0);
  const int e0 = blockIdx.x * epc;
  uint8_t* xsm = dsm_dec;                                                          // [tn][NC] chunks
  float* part = reinterpret_cast<float*>(dsm_dec + (size_t)tpc * NC * kDecPitch);  // [epc][tpc][NC + 1]
  const int c = threadIdx.x % NC;
  const int g = threadIdx.x / NC;
  // this thread's experts and their Wr chunks, loaded once (all loads in flight together)
  uint4 wv[EPT][8];
  bool has[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int el = g * EPT + j;
    has[j] = el < epc && e0 + el < E;
    const uint4* wp = reinterpret_cast<const uint4*>(wr + (size_t)(has[j] ? e0 + el : 0) * H + (size_t)c * kRouterChunk);
#pragma unroll
    for (int i = 0; i < 8; ++i) wv[j][i] = has[j] ? __ldg(wp + i) : make_uint4(0, 0, 0, 0);
  }
  // stage the block's rows: 16-byte unit u of chunk (t, c) from x[t0 + t, 64 c + 8 u]
  for (int i = threadIdx.x; i < tn * NC * 8; i += blockDim.x) {
    const int u = i & 7, tc = i >> 3;
    const int t = tc / NC, cc = tc - t * NC;
    cp_async_16(xsm + (size_t)tc * kDecPitch + u * 16, x + (size_t)(t0 + t) * H + cc * kRouterChunk + u * 8, 16);
  }
  cp_async_wait_all();
  __syncthreads();
  // two tokens per pass: independent chains, each in element order from +0
  for (int t = 0; t < tn; t += 2) {
    const bool two = t + 1 < tn;
    const uint4* xp0 = reinterpret_cast<const uint4*>(xsm + ((size_t)t * NC + c) * kDecPitch);
    const uint4* xp1 = reinterpret_cast<const uint4*>(xsm + ((size_t)(two ? t + 1 : t) * NC + c) * kDecPitch);
    float p0[EPT], p1[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) p0[j] = p1[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 a = xp0[i];
      const uint4 b = xp1[i];
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        p0[j] = fma2_bf16(a.x, wv[j][i].x, p0[j]);
        p1[j] = fma2_bf16(b.x, wv[j][i].x, p1[j]);
        p0[j] = fma2_bf16(a.y, wv[j][i].y, p0[j]);
        p1[j] = fma2_bf16(b.y, wv[j][i].y, p1[j]);
        p0[j] = fma2_bf16(a.z, wv[j][i].z, p0[j]);
        p1[j] = fma2_bf16(b.z, wv[j][i].z, p1[j]);
        p0[j] = fma2_bf16(a.w, wv[j][i].w, p0[j]);
        p1[j] = fma2_bf16(b.w, wv[j][i].w, p1[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      if (!has[j]) continue;
      float* pp = part + ((size_t)(g * EPT + j) * tpc + t) * (NC + 1) + c;
      pp[0] = p0[j];
      if (two) pp[NC + 1] = p1[j];
    }
  }
  // MXFP8 quantisation of this token block's rows: the CTAs of the block take the 32-blocks in turn
  if (xq) {
    const int nblk = tn * H / 32;
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += gridDim.x * blockDim.x) {
      const int t = b / (H / 32), h = (b % (H / 32)) * 32;
      const uint4* src = reinterpret_cast<const uint4*>(xsm + ((size_t)t * NC + h / kRouterChunk) * kDecPitch +
                                                        (h % kRouterChunk) * 2);
      float f[32];
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = src[i];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f[8 * i + 2 * q] = bf_lo(w4[q]);
          f[8 * i + 2 * q + 1] = bf_hi(w4[q]);
          m = fmaxf(m, fmaxf(fabsf(f[8 * i + 2 * q]), fabsf(f[8 * i + 2 * q + 1])));
        }
      }
      const int se = e4m3_scale_exp(m);
      const float sc = pow2_neg(se);
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        o[i] = e4m3x2(f[4 * i] * sc, f[4 * i + 1] * sc) | (e4m3x2(f[4 * i + 2] * sc, f[4 * i + 3] * sc) << 16);
      uint4* dq = reinterpret_cast<uint4*>(xq + (size_t)(t0 + t) * H + h);
      dq[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dq[1] = make_uint4(o[4], o[5], o[6], o[7]);
      xs[(size_t)(t0 + t) * (H / 32) + h / 32] = (uint8_t)(se + 127);
    }
  }
  __syncthreads();
  for (int it = threadIdx.x; it < epc * tn; it += blockDim.x) {
    const int el = it / tn, t = it - el * tn;
    const int e = e0 + el;
    if (e >= E) continue;
    const float* pp = part + ((size_t)el * tpc + t) * (NC + 1);
    float acc = 0.f;
    for (int cc = 0; cc < NC; ++cc) acc = __fadd_rn(acc, pp[cc]);
    const float sc = sigmoid_cw(acc);
    const float ky = __fadd_rn(sc, bias[e]);
    score[(size_t)(t0 + t) * E + e] = sc;
    key[(size_t)(t0 + t) * E + e] = ky;
    // the self-routing GEMM's copies of the (key, score) pairs (nullable)
    if (sel)
      for (int r = 0; r < kSelfPlanReplicas; ++r) sel[((size_t)r * T + t0 + t) * E + e] = make_float2(ky, sc);
  }
}

// ---------------------------------------------------------------------------------------------
// Logits, large T: 64 tokens x 64 experts per CTA, 4 x 4 outputs per thread, one 64-wide h chunk
// per shared-memory stage, staged transposed ([h][token], [h][expert]) so that each h step is two
// 16-byte shared loads and 16 fma. Each output keeps its chunk partial (sequential fma from +0
// over the chunk) and adds it to its running sum after the chunk: the same order as the small-T
// kernels.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) router_tiled_kernel(const uint16_t* __restrict__ x,
                                                           const uint16_t* __restrict__ wr,
                                                           const float* __restrict__ bias, int T, int H, int E,
                                                           float* __restrict__ score, float* __restrict__ key) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) float xs[kRouterChunk][64];
  __shared__ __align__(16) float ws[kRouterChunk][64];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
  // staging: thread -> (row = tid % 64, 16 consecutive h); a warp stores 32 rows of one h
  const int srow = tid & 63, sh = (tid >> 6) * 16;
  float acc[4][4], part[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int h0 = 0; h0 < H; h0 += kRouterChunk) {
    __syncthreads();
    {
      uint4 xa = make_uint4(0, 0, 0, 0), xb = xa, wa = xa, wb = xa;
      if (t0 + srow < T) {
        const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)(t0 + srow) * H + h0 + sh);
        xa = __ldg(xp);
        xb = __ldg(xp + 1);
      }
      if (e0 + srow < E) {
        const uint4* wp = reinterpret_cast<const uint4*>(wr + (size_t)(e0 + srow) * H + h0 + sh);
        wa = __ldg(wp);
        wb = __ldg(wp + 1);
      }
      const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      const uint32_t ww[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        xs[sh + 2 * q][srow] = bf_lo(xw[q]);
        xs[sh + 2 * q + 1][srow] = bf_hi(xw[q]);
        ws[sh + 2 * q][srow] = bf_lo(ww[q]);
        ws[sh + 2 * q + 1][srow] = bf_hi(ww[q]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) part[i][j] = 0.f;
#pragma unroll 8
    for (int h = 0; h < kRouterChunk; ++h) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[h][4 * ty]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[h][4 * tx]);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = __fmaf_rn(xa[i], wa[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = __fadd_rn(acc[i][j], part[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + 4 * ty + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + 4 * tx + j;
      if (e >= E) continue;
      const float sc = sigmoid_cw(acc[i][j]);
      score[(size_t)t * E + e] = sc;
      key[(size_t)t * E + e] = __fadd_rn(sc, bias[e]);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Top-k + plan. Each warp routes its tokens one at a time: k rounds of a warp arg-max over
// (key descending, expert ascending). A CTA then builds, per expert, a bitmask of its block's
// live tokens that chose it: the rank of a slot inside its expert is the number of lower token
// bits set, so the plan order inside an expert is token order, with no atomics whose order
// matters. With a single block (T <= kPlanBlock) one CTA also scans and scatters the plan.
// ---------------------------------------------------------------------------------------------

__device__ void block_exclusive_scan(int* vals, int n, int* total) {
  // vals in shared memory, n <= 1024; blockDim.x == 512
  __shared__ int tmp[1024];
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) tmp[i] = i < n ? vals[i] : 0;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    int v[2];
    for (int q = 0; q < 2; ++q) {
      int i = threadIdx.x + q * 512;
      v[q] = (i >= off) ? tmp[i - off] : 0;
    }
    __syncthreads();
    for (int q = 0; q < 2; ++q) tmp[threadIdx.x + q * 512] += v[q];
    __syncthreads();
  }
  // tmp is now the inclusive scan
  for (int i = threadIdx.x; i < n; i += blockDim.x) vals[i] = i == 0 ? 0 : tmp[i - 1];
  if (threadIdx.x == 0) *total = n > 0 ? tmp[n - 1] : 0;
  __syncthreads();
}

// Exclusive scan of vals[0..n) in shared memory by the whole block (any multiple of 32 threads):
// each thread sums a contiguous segment, a two-level warp scan gives the segment offsets, each
// thread rewrites its segment. *total = the sum. wsum: 32 ints of shared scratch.
__device__ void block_scan_segments(int* vals, int n, int* total, int* wsum) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
  const int c = (n + nt - 1) / nt;
  const int b = min(n, tid * c), e = min(n, b + c);
  int s = 0;
  for (int i = b; i < e; ++i) s += vals[i];
  int x = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) wsum[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < nw) wsum[lane] = w;
  }
  __syncthreads();
  int base = (wid > 0 ? wsum[wid - 1] : 0) + x - s;
  for (int i = b; i < e; ++i) {
    const int v = vals[i];
    vals[i] = base;
    base += v;
  }
  if (tid == 0) *total = wsum[nw - 1];
  __syncthreads();
}

// Anchored verify rows (TP4 serving profile README, settings table row "Verify length"): a row
// with anchor[t] = a reuses row a's experts (a routes itself) and weights them with its own scores,
// so it reaches no expert its anchor does not. An anchor outside [0, T) or one that is itself
// anchored is ignored (the row routes itself) and recorded in the status word.
__device__ __forceinline__ int anchor_of(const int32_t* __restrict__ anchor, int t, int T, uint32_t* status) {
  if (!anchor) return -1;
  const int a = anchor[t];
  if (a < 0) return -1;
  if (a >= T || anchor[a] != -1) {
    if (status) atomicCAS(status, 0u, (uint32_t)DEV_BAD_INPUT);
    return -1;
  }
  return a;
}

// Lane j < k gets expert e (the anchor's j-th choice) and the row's weight score[e] / sum, the sum
// taken in rank order (identical on every lane).
__device__ __forceinline__ void anchored_weights(const float* __restrict__ srow, int e, int k, int lane, float* w) {
  const float sc = lane < k ? __ldcg(srow + e) : 0.f;
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, sc, j));
  *w = __fdiv_rn(sc, sum);
}

// Top-k alone, one warp per token over the whole grid (the plan kernels read its result when the
// rows outnumber one plan CTA's warps).
template <int NI>
__global__ void __launch_bounds__(256) topk_select_kernel(const float* __restrict__ score,
                                                          const float* __restrict__ key, int T, int E, int k,
                                                          int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w,
                                                          const int32_t* __restrict__ anchor, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    if (anchor_of(anchor, t, T, status) >= 0) continue;      // filled in by anchor_fixup_kernel
    int my_e = -1;
    float my_s = 0.f, sum = 0.f;
    warp_topk<NI>(key + (size_t)t * E, score + (size_t)t * E, E, k, lane, nullptr, &my_e, &my_s, &sum);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_e;
      topk_w[(size_t)t * k + lane] = __fdiv_rn(my_s, sum);
    }
  }
}

// Anchored rows of the grid-wide selection: one warp per row copies the anchor's choices.
__global__ void __launch_bounds__(256) anchor_fixup_kernel(const float* __restrict__ score, int T, int E, int k,
                                                           const int32_t* __restrict__ anchor,
                                                           int32_t* __restrict__ topk_idx,
                                                           float* __restrict__ topk_w) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    const int a = anchor_of(anchor, t, T, nullptr);
    if (a < 0) continue;
    const int e = lane < k ? topk_idx[(size_t)a * k + lane] : 0;
    float w;
    anchored_weights(score + (size_t)t * E, e, k, lane, &w);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = e;
      topk_w[(size_t)t * k + lane] = w;
    }
  }
}

// Top-k and the whole plan for T <= kPlanBlock rows in one CTA (any multiple of 32 threads, one
// token per warp at a time): selection (self-routed rows, then anchored rows), per-expert token
// bitmasks (plan order inside an expert = token order), counts, offsets, scatter. Without
// kSelect the choices come from topk_idx (written by topk_select_kernel; no anchors).
// Shared scratch: mask [E * 8] u32, sidx [kPlanBlock * k] i16, scnt [E] i32, wsum [32] i32, total.
template <int NI, bool kSelect = true>
__device__ void plan_single_block(const float* __restrict__ score, const float* __restrict__ key,
                                  const uint8_t* __restrict__ dead, int T, int E, int k, int32_t* __restrict__ topk_idx,
                                  float* __restrict__ topk_w, int32_t* __restrict__ counts,
                                  int32_t* __restrict__ offsets, int32_t* __restrict__ slot_of_row,
                                  int32_t* __restrict__ row_of_slot, const int32_t* __restrict__ anchor,
                                  uint32_t* status, uint32_t* mask, int16_t* sidx, int* scnt, int* wsum, int* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (!kSelect)
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) sidx[i] = (int16_t)__ldcg(topk_idx + i);
  for (int t = warp; kSelect && t < T; t += nwarps) {
    if (anchor_of(anchor, t, T, status) >= 0) continue;      // after every self-routed row
    int my_e = -1;
    float my_s = 0.f, sum = 0.f;
    warp_topk<NI>(key + (size_t)t * E, score + (size_t)t * E, E, k, lane, sidx + t * k, &my_e, &my_s, &sum);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_e;
      topk_w[(size_t)t * k + lane] = __fdiv_rn(my_s, sum);
    }
  }
  // the bitmasks are first used after the barrier below: zeroed after the selection, off its path
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) mask[i] = 0;
  if (anchor) {
    __syncthreads();
    for (int t = warp; t < T; t += nwarps) {
      const int a = anchor_of(anchor, t, T, nullptr);
      if (a < 0) continue;
      const int e = lane < k ? (int)sidx[a * k + lane] : 0;
      float w;
      anchored_weights(score + (size_t)t * E, e, k, lane, &w);
      if (lane < k) {
        topk_idx[(size_t)t * k + lane] = e;
        topk_w[(size_t)t * k + lane] = w;
        sidx[t * k + lane] = (int16_t)e;
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int t = i / k;
    if (dead && dead[t]) {
      sidx[i] = -1;                                          // dead slot: no plan row
      continue;
    }
    atomicOr(&mask[sidx[i] * 8 + (t >> 5)], 1u << (t & 31));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) c += __popc(mask[e * 8 + w]);
    scnt[e] = c;
    counts[e] = c;
  }
  __syncthreads();
  block_scan_segments(scnt, E, total, wsum);
  for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = scnt[e];
  if (threadIdx.x == 0) offsets[E] = *total;
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int t = i / k;
    const int e = sidx[i];
    if (e < 0) {
      row_of_slot[i] = -1;
      continue;
    }
    const int w = t >> 5;
    int r = 0;
    for (int q = 0; q < w; ++q) r += __popc(mask[e * 8 + q]);
    r += __popc(mask[e * 8 + w] & ((1u << (t & 31)) - 1u));
    const int p = scnt[e] + r;
    slot_of_row[p] = i;
    row_of_slot[i] = p;
  }
}

inline size_t plan_single_smem(int E, int k) {
  return align_up((size_t)E * 8 * 4, 16) + align_up((size_t)kPlanBlock * k * 2, 16) + align_up((size_t)E * 4, 16) +
         32 * 4 + 16;
}

// T <= kPlanBlock: top-k and plan in one CTA.
// Threads of the one-CTA plan: a warp selects one row at a time, so more warps take more rows at
// once; up to 8 keys per lane (E <= 256) the registers allow 32 warps. Small batches launch 8 warps
// (every later step of the plan meets at block-wide barriers, cheaper with fewer warps).
template <int NI>
constexpr int plan_single_threads() { return NI <= 8 ? 1024 : 512; }
template <int NI>
inline int plan_single_launch_threads(int T) { return (NI <= 8 && T <= 8) ? 256 : plan_single_threads<NI>(); }

template <int NI, bool kSelect = true>
__global__ void __launch_bounds__(plan_single_threads<NI>()) topk_plan_single_kernel(const float* __restrict__ score,
                                                               const float* __restrict__ key,
                                                               const uint8_t* __restrict__ dead, int T, int E, int k,
                                                               int32_t* __restrict__ topk_idx,
                                                               float* __restrict__ topk_w,
                                                               int32_t* __restrict__ counts,
                                                               int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ slot_of_row,
                                                               int32_t* __restrict__ row_of_slot,
                                                               const int32_t* __restrict__ anchor, uint32_t* status,
                                                               uint32_t* __restrict__ ready) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) uint8_t psm[];
  uint32_t* mask = reinterpret_cast<uint32_t*>(psm);
  int16_t* sidx = reinterpret_cast<int16_t*>(psm + align_up((size_t)E * 8 * 4, 16));
  int* scnt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(sidx) + align_up((size_t)kPlanBlock * k * 2, 16));
  int* wsum = scnt + align_up((size_t)E * 4, 16) / 4;
  int* total = wsum + 32;
  plan_single_block<NI, kSelect>(score, key, dead, T, E, k, topk_idx, topk_w, counts, offsets, slot_of_row,
                                 row_of_slot, anchor, status, mask, sidx, scnt, wsum, total);
  // tile counters of the one-launch W13 + W2 GEMM (E per expert + 1 total; nullable): zero them
  // (that GEMM reads them only after this grid has completed)
  if (ready)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) ready[e] = 0;
}

// Multi-block plan, step 1: one CTA per kPlanBlock tokens reads the choices from topk_idx (written
// by topk_select_kernel / anchor_fixup_kernel) and writes its per-expert counts and each slot's
// rank inside its expert (the number of lower token bits set in the block's bitmask).
__global__ void __launch_bounds__(512) topk_plan_kernel(const uint8_t* __restrict__ dead, int T, int E, int k,
                                                        const int32_t* __restrict__ topk_idx,
                                                        int32_t* __restrict__ cnt, int32_t* __restrict__ rank) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t dsm[];
  uint32_t* mask = dsm;                                         // [E][8]
  int16_t* sidx = reinterpret_cast<int16_t*>(dsm + E * 8);      // [kPlanBlock][k]
  const int tb0 = blockIdx.x * kPlanBlock;
  const int nt = min(kPlanBlock, T - tb0);
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) mask[i] = 0;
  for (int i = threadIdx.x; i < nt * k; i += blockDim.x) sidx[i] = (int16_t)topk_idx[(size_t)tb0 * k + i];
  __syncthreads();
  // per-expert token bitmasks of this block (bit order = token order)
  for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
    const int tl = i / k;
    if (dead && dead[tb0 + tl]) continue;
    atomicOr(&mask[sidx[i] * 8 + (tl >> 5)], 1u << (tl & 31));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) c += __popc(mask[e * 8 + w]);
    cnt[(size_t)blockIdx.x * E + e] = c;
  }
  for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
    const int tl = i / k;
    const int t = tb0 + tl;
    int r = -1;
    if (!(dead && dead[t])) {
      const int e = sidx[i];
      const int w = tl >> 5;
      r = 0;
      for (int q = 0; q < w; ++q) r += __popc(mask[e * 8 + q]);
      r += __popc(mask[e * 8 + w] & ((1u << (tl & 31)) - 1u));
    }
    rank[(size_t)t * k + (i % k)] = r;
  }
}

// Multi-block plan, step 2 (one CTA): per-expert totals, offsets, and each block's base row.
__global__ void __launch_bounds__(512) plan_scan_kernel(const int32_t* __restrict__ cnt, int nb, int E,
                                                        int32_t* __restrict__ base, int32_t* __restrict__ counts,
                                                        int32_t* __restrict__ offsets, uint32_t* __restrict__ ready) {
  pdl_trigger();
  pdl_wait();
  if (ready)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) ready[e] = 0;
  __shared__ int tot[kMaxE];
  __shared__ int total_s;
  constexpr int U = 8;                            // block counts loaded per step (all in flight)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += U) {
      int c[U];
#pragma unroll
      for (int j = 0; j < U; ++j) c[j] = b0 + j < nb ? cnt[(size_t)(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < U; ++j) run += c[j];
    }
    tot[e] = run;
    counts[e] = run;
  }
  __syncthreads();
  block_exclusive_scan(tot, E, &total_s);
  for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = tot[e];
  if (threadIdx.x == 0) offsets[E] = total_s;
  // base[b][e] = offset of expert e + rows of e in blocks before b
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = tot[e];
    for (int b0 = 0; b0 < nb; b0 += U) {
      int c[U];
#pragma unroll
      for (int j = 0; j < U; ++j) c[j] = b0 + j < nb ? cnt[(size_t)(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < U; ++j) {
        if (b0 + j < nb) base[(size_t)(b0 + j) * E + e] = run;
        run += c[j];
      }
    }
  }
}

// Multi-block plan, step 3: scatter every live slot to its plan row.
__global__ void plan_scatter_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ rank,
                                    const int32_t* __restrict__ base, int T, int E, int k,
                                    int32_t* __restrict__ slot_of_row, int32_t* __restrict__ row_of_slot) {
  pdl_trigger();
  pdl_wait();
  const long long n = (long long)T * k;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int r = rank[i];
    if (r < 0) { row_of_slot[i] = -1; continue; }
    const int t = (int)(i / k);
    const int b = t / kPlanBlock;
    const int e = topk_idx[i];
    const int p = base[(size_t)b * E + e] + r;
    slot_of_row[p] = (int)i;
    row_of_slot[i] = p;
  }
}

template <int NI>
static int launch_topk_plan_ni(int nb, int E, size_t smem, cudaStream_t st, const float* score, const float* key,
                               const uint8_t* dead, int T, int k, int32_t* topk_idx, float* topk_w, int32_t* cnt,
                               int32_t* rank, int32_t* counts, int32_t* offsets, int32_t* slot_of_row,
                               int32_t* row_of_slot, const int32_t* anchor, uint32_t* status, uint32_t* ready) {
  if (ensure_smem_limit((const void*)topk_plan_single_kernel<NI>, 64 * 1024) ||
      ensure_smem_limit((const void*)topk_plan_single_kernel<NI, false>, 64 * 1024) ||
      ensure_smem_limit((const void*)topk_plan_kernel, 64 * 1024))
    return MOE_ERR_CUDA;
  if (nb == 1 && !anchor && T > std::min(24, plan_single_threads<NI>() / 32)) {
    // many rows for the plan CTA's warps (at 32 rows its one round of selections already contend
    // for one SM): the selection runs on the whole GPU (one warp per row, all rows at once) and
    // the one CTA only plans from its lists
    const int sel_blocks = (int)std::min<long long>(((long long)T + 7) / 8, (long long)num_sms() * 8);
    const int rc = launch_pdl(topk_select_kernel<NI>, dim3(sel_blocks), dim3(256), 0, st, score, key, T, E, k,
                              topk_idx, topk_w, anchor, status);
    if (rc) return rc;
    return launch_pdl(topk_plan_single_kernel<NI, false>, dim3(1), dim3(plan_single_launch_threads<NI>(T)),
                      plan_single_smem(E, k), st, score, key, dead, T, E, k, topk_idx, topk_w, counts, offsets,
                      slot_of_row, row_of_slot, anchor, status, ready);
  }
  if (nb == 1)
    return launch_pdl(topk_plan_single_kernel<NI>, dim3(1), dim3(plan_single_launch_threads<NI>(T)),
                      plan_single_smem(E, k),
                      st, score, key, dead, T,
                      E, k, topk_idx, topk_w, counts, offsets, slot_of_row, row_of_slot, anchor, status, ready);
  // many blocks: selection spread over the whole GPU (anchored rows next), then the per-block plan
  const int sel_blocks = (int)std::min<long long>(((long long)T + 7) / 8, (long long)num_sms() * 8);
  int rc = launch_pdl(topk_select_kernel<NI>, dim3(sel_blocks), dim3(256), 0, st, score, key, T, E, k, topk_idx,
                      topk_w, anchor, status);
  if (rc) return rc;
  if (anchor) {
    rc = launch_pdl(anchor_fixup_kernel, dim3(sel_blocks), dim3(256), 0, st, score, T, E, k, anchor, topk_idx, topk_w);
    if (rc) return rc;
  }
  return launch_pdl(topk_plan_kernel, dim3(nb), dim3(512), smem, st, dead, T, E, k, (const int32_t*)topk_idx, cnt,
                    rank);
}

// NI = experts per lane, the smallest power of two with 32 * NI >= E.
static int launch_topk_plan(int nb, int E, size_t smem, cudaStream_t st, const float* score, const float* key,
                            const uint8_t* dead, int T, int k, int32_t* topk_idx, float* topk_w, int32_t* cnt,
                            int32_t* rank, int32_t* counts, int32_t* offsets, int32_t* slot_of_row,
                            int32_t* row_of_slot, const int32_t* anchor, uint32_t* status, uint32_t* ready) {
#define MOE_TOPK_CASE(N)                                                                                        \
  if (E <= 32 * N)                                                                                              \
    return launch_topk_plan_ni<N>(nb, E, smem, st, score, key, dead, T, k, topk_idx, topk_w, cnt, rank, counts, \
                                  offsets, slot_of_row, row_of_slot, anchor, status, ready);
  MOE_TOPK_CASE(1)
  MOE_TOPK_CASE(2)
  MOE_TOPK_CASE(4)
  MOE_TOPK_CASE(8)
  MOE_TOPK_CASE(16)
  MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
  return MOE_ERR_UNSUPPORTED_SHAPE;
}

// One plan block, plain launch (no programmatic serialisation): used by the allocation-free router.
template <int NI>
static int launch_topk_single_plain_ni(cudaStream_t st, const float* score, const float* key, const uint8_t* dead,
                                       int T, int E, int k, int32_t* topk_idx, float* topk_w, int32_t* counts,
                                       int32_t* offsets, int32_t* slot_of_row, int32_t* row_of_slot) {
  if (ensure_smem_limit((const void*)topk_plan_single_kernel<NI>, 64 * 1024)) return MOE_ERR_CUDA;
  topk_plan_single_kernel<NI><<<1, plan_single_launch_threads<NI>(T), plan_single_smem(E, k), st>>>(score, key, dead,
                                                                                                   T, E, k,
                                                                                          topk_idx, topk_w,
                                                                       counts, offsets, slot_of_row, row_of_slot,
                                                                       nullptr, nullptr, nullptr);
  return launch_status();
}

static int launch_topk_single_plain(int E, cudaStream_t st, const float* score, const float* key,
                                    const uint8_t* dead, int T, int k, int32_t* topk_idx, float* topk_w,
                                    int32_t* counts, int32_t* offsets, int32_t* slot_of_row, int32_t* row_of_slot) {
#define MOE_TOPK_CASE(N)                                                                                          \
  if (E <= 32 * N)                                                                                                \
    return launch_topk_single_plain_ni<N>(st, score, key, dead, T, E, k, topk_idx, topk_w, counts, offsets,      \
                                          slot_of_row, row_of_slot);
  MOE_TOPK_CASE(1)
  MOE_TOPK_CASE(2)
  MOE_TOPK_CASE(4)
  MOE_TOPK_CASE(8)
  MOE_TOPK_CASE(16)
  MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
  return MOE_ERR_UNSUPPORTED_SHAPE;
}

static bool decode_router_fits(int T, int H, int E) {
  const DecodeRouterCfg dc = decode_router_cfg(T, H, E);
  return T <= kDecMaxT && dc.threads <= kDecThreadsMax && dc.smem <= kDecodeSmemMax;
}

// The decode router (decode_router_fits): scores and keys, plus xq/xs, the zeroed counters in
// ready and the (key, score) copies in sel when those are non-null.
static int launch_router_decode(const moe_shape* s, const uint16_t* x, const uint16_t* wr, const float* bias,
                                float* score, float* key, uint8_t* xq, uint8_t* xs, uint32_t* ready, float2* sel,
                                cudaStream_t st) {
  const int T = s->T, E = s->E, H = s->H;
  const DecodeRouterCfg dc = decode_router_cfg(T, H, E);
  const dim3 grid(ceil_div(E, dc.epc), ceil_div(T, dc.tpc));
  if (dc.ept == 1) {
    if (ensure_smem_limit((const void*)router_decode_kernel<1>, (int)kDecodeSmemMax)) return MOE_ERR_CUDA;
    return launch_pdl(router_decode_kernel<1>, grid, dim3(dc.threads), dc.smem, st, x, wr, bias, T, H, E, dc.epc,
                      dc.tpc, score, key, xq, xs, ready, sel);
  }
  if (ensure_smem_limit((const void*)router_decode_kernel<2>, (int)kDecodeSmemMax)) return MOE_ERR_CUDA;
  return launch_pdl(router_decode_kernel<2>, grid, dim3(dc.threads), dc.smem, st, x, wr, bias, T, H, E, dc.epc,
                    dc.tpc, score, key, xq, xs, ready, sel);
}

bool self_plan_supported(const moe_shape* s) {
  return s->T >= 1 && s->T <= kSelfPlanMaxT && s->E <= kSelfPlanMaxE && fused_gemms_supported(s) &&
         decode_router_fits(s->T, s->H, s->E);
}

int launch_router_decode_scores(const moe_shape* s, const uint16_t* x, const uint16_t* wr, const float* bias, void* ws,
                                cudaStream_t st, uint8_t* xq, uint8_t* xs, uint32_t* ready) {
  if (!self_plan_supported(s) || !xq || !xs || !ready) return MOE_ERR_UNSUPPORTED_SHAPE;
  const Workspace L = workspace_layout(s);
  return launch_router_decode(s, x, wr, bias, ws_ptr<float>(ws, L.score), ws_ptr<float>(ws, L.key), xq, xs, ready,
                              ws_ptr<float2>(ws, L.selrep), st);
}

int launch_route(const moe_shape* s, const uint16_t* x, const uint16_t* wr, const float* bias, const uint8_t* dead,
                 int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets, int32_t* slot_of_row,
                 int32_t* row_of_slot, void* ws, cudaStream_t st, uint8_t* xq, uint8_t* xs, bool* quant_done,
                 const int32_t* anchor, uint32_t* ready) {
  if (quant_done) *quant_done = false;
  const Workspace L = workspace_layout(s);
  const int T = s->T, E = s->E, k = s->k, H = s->H;
  if (T == 0) {
    cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st);
    cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    return launch_status();
  }
  float* score = ws_ptr<float>(ws, L.score);
  float* key = ws_ptr<float>(ws, L.key);
  int rc0 = MOE_OK;
  if (decode_router_fits(T, H, E)) {
    const bool fuse = xq && xs;
    rc0 = launch_router_decode(s, x, wr, bias, score, key, fuse ? xq : nullptr, fuse ? xs : nullptr, nullptr, nullptr,
                               st);
    if (quant_done) *quant_done = fuse;
  } else if (T <= kSmallT) {
    rc0 = launch_pdl(router_small_kernel, dim3(ceil_div(E, 8)), dim3(256), 0, st, x, wr, bias, T, H, E, score, key);
  } else if (router_screen_supported(s)) {
    rc0 = launch_router_screen(s, x, wr, bias, ws, score, key, st, anchor);
  } else {
    rc0 = launch_pdl(router_tiled_kernel, dim3(ceil_div(T, 64), ceil_div(E, 64)), dim3(256), 0, st, x, wr, bias, T,
                     H, E, score, key);
  }
  int rc = rc0;
  if (rc) return rc;
  const int nb = ceil_div(T, kPlanBlock);
  const size_t smem = (size_t)E * 8 * 4 + (size_t)kPlanBlock * k * 2;
  int32_t* cnt = ws_ptr<int32_t>(ws, L.cnt);
  int32_t* base = ws_ptr<int32_t>(ws, L.base);
  int32_t* rank = ws_ptr<int32_t>(ws, L.rank);
  rc = launch_topk_plan(nb, E, smem, st, score, key, dead, T, k, topk_idx, topk_w, cnt, rank, counts, offsets,
                        slot_of_row, row_of_slot, anchor, ws_ptr<uint32_t>(ws, L.status), ready);
  if (rc || nb == 1) return rc;
  rc = launch_pdl(plan_scan_kernel, dim3(1), dim3(512), 0, st, cnt, nb, E, base, counts, offsets, ready);
  if (rc) return rc;
  const long long n = (long long)T * k;
  const int blocks = (int)std::min<long long>((n + 255) / 256, (long long)num_sms() * 4);
  return launch_pdl(plan_scatter_kernel, dim3(blocks), dim3(256), 0, st, topk_idx, rank, base, T, E, k, slot_of_row,
                    row_of_slot);
}

// ---------------------------------------------------------------------------------------------
// Combine: out[t] = bf16_rne(((y_0 + y_1) + ...) + y_{k-1}) in fp32, slots in rank order, where
// y_j = topk_w[t, j] * y[row_of_slot[t k + j]] (one fp32 rounding: the down projection's plan-order
// rows arrive before their routing weight); then + y_shared[t] when a shared expert ran. Rows
// without live slots, and rows the caller's dead mask flags, get +0.0 (a flagged row that still
// holds slots is recorded in the status word). 8 hidden elements per thread.
// ---------------------------------------------------------------------------------------------
__global__ void combine_kernel(const float* __restrict__ y, const float* __restrict__ topk_w,
                               const int32_t* __restrict__ row_of_slot, int T, int H, int k,
                               uint16_t* __restrict__ out, const float* __restrict__ y_shared,
                               const uint8_t* __restrict__ dead, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int H8 = H / 8;
  const long long n = (long long)T * H8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    combine_unit<false>(y, topk_w, row_of_slot, (int)(i / H8), (int)(i % H8), H, k, out, y_shared, dead, status);
}

int launch_combine(const moe_shape* s, const float* y, const float* topk_w, const int32_t* row_of_slot,
                   uint16_t* out, cudaStream_t st, const float* y_shared, const uint8_t* dead, uint32_t* status) {
  const long long n = (long long)s->T * (s->H / 8);
  if (n == 0) return MOE_OK;
  const int blocks = (int)std::min<long long>((n + 255) / 256, (long long)num_sms() * 8);
  return launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, st, y, topk_w, row_of_slot, s->T, s->H, s->k, out,
                    y_shared, dead, status);
}

}  // namespace moe

using namespace moe;

extern "C" int moe_route_topk(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* bias,
                              const uint8_t* dead, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                              int32_t* expert_offsets, int32_t* slot_of_row, int32_t* row_of_slot, void* ws,
                              size_t ws_bytes, void* stream) {
  return moe_route_topk_anchored(s, x, w_router, bias, dead, nullptr, topk_idx, topk_w, expert_counts,
                                 expert_offsets, slot_of_row, row_of_slot, ws, ws_bytes, stream);
}

extern "C" int moe_route_topk_anchored(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
                                       const float* bias, const uint8_t* dead, const int32_t* anchor,
                                       int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                                       int32_t* expert_offsets, int32_t* slot_of_row, int32_t* row_of_slot, void* ws,
                                       size_t ws_bytes, void* stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (anchor && (reinterpret_cast<uintptr_t>(anchor) & 3)) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && (!x || !w_router || !bias || !topk_idx || !topk_w || !slot_of_row || !row_of_slot))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(w_router) & 15))
    return MOE_ERR_INVALID_ARG;
  int rc = ws_check(s, ws, ws_bytes);
  if (rc) return rc;
  return launch_route(s, x, w_router, bias, dead, topk_idx, topk_w, expert_counts, expert_offsets, slot_of_row,
                      row_of_slot, ws, static_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, anchor, nullptr);
}

// ---------------------------------------------------------------------------------------------
// Allocation-free router entry point.
//
// Some callers cannot hand this library a workspace: a serving engine that reserved all of HBM
// for its own pool at start-up has no bytes left for a cudaMalloc, and code running inside a host
// framework's custom-op or callback may be forbidden from allocating at all. For them the router
// keeps its scratch (sigmoid scores and selection keys, 4 bytes each per (row, expert)) in this
// file-scope device array instead of the caller's workspace. Every GPU that loads the library
// holds the array (512 KiB) until the process exits. All calls share it, so calls that may overlap
// on the GPU (different streams, or different host threads) race on it; callers must serialise
// them. Each call writes every scratch element it reads before reading it, so nothing needs to be
// cleared between calls.
// ---------------------------------------------------------------------------------------------
namespace moe {
constexpr int kNoAllocMaxRowsTimesExperts = 65536;        // T * E limit (and T <= kPlanBlock)
static __device__ __align__(256) float g_route_scratch[2 * kNoAllocMaxRowsTimesExperts];
}  // namespace moe

#include <mutex>

extern "C" int moe_route_topk_noalloc(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
                                      const float* bias, const uint8_t* dead, int32_t* topk_idx, float* topk_w,
                                      int32_t* expert_counts, int32_t* expert_offsets, int32_t* slot_of_row,
                                      int32_t* row_of_slot, void* stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->T > kPlanBlock || (int64_t)s->T * s->E > kNoAllocMaxRowsTimesExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && (!x || !w_router || !bias || !topk_idx || !topk_w || !slot_of_row || !row_of_slot))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(w_router) & 15))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = s->T, E = s->E, k = s->k, H = s->H;
  if (T == 0) {
    if (cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, st) != cudaSuccess ||
        cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  // Set-up, once per device and with that device current: the host-side name of the array is
  // not a device address, so ask the runtime for it.
  static std::mutex mu;
  static float* scratch_of_device[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  float* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!scratch_of_device[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
      scratch_of_device[dev] = static_cast<float*>(p);
    }
    scratch = scratch_of_device[dev];
  }
  float* score = scratch;
  float* key = scratch + (size_t)T * E;
  if (T <= kSmallT) {
    router_small_kernel<<<ceil_div(E, 8), 256, 0, st>>>(x, w_router, bias, T, H, E, score, key);
  } else {
    dim3 grid(ceil_div(T, 64), ceil_div(E, 64));
    router_tiled_kernel<<<grid, 256, 0, st>>>(x, w_router, bias, T, H, E, score, key);
  }
  int rc = launch_status();
  if (rc) return rc;
  // one plan block (T <= kPlanBlock): the kernel scans and scatters itself and never touches the
  // multi-block count/rank arrays
  rc = launch_topk_single_plain(E, st, score, key, dead, T, k, topk_idx, topk_w, expert_counts, expert_offsets,
                                slot_of_row, row_of_slot);
  if (rc) return rc;
  return launch_status();
}
