// Certified tensor-core screen for the router at large T, followed by an exact recompute of the
// few experts that can still be in a row's top-k. The selected experts, their weights and the
// plan are bit-identical to the fixed-order fp32 router (the screen only prunes experts that
// provably cannot be selected).
//
// "New Deepseek 4.1 flash recipe", post 6 "How it works" item 3 (TileKernels MoE top-k gate) and
// "Why TileLang" (fixed-order reductions); TP4 serving profile README, settings table, "Target LM
// head" row: read a cheap screen with a proven error bound, then compute exactly only what can
// still win.
//
// 1. router_norms_kernel: ||x_t||_2 and ||Wr_e||_2 (fp32, rounded up by a relative 2^-10).
// 2. router_screen_kernel: L~ = x Wr^T on tcgen05 (bf16 x bf16, fp32 accumulate; 128 rows x all
//    E experts per CTA, TMA-fed, accumulator in TMEM). bf16 products are exact, so the only error
//    is accumulation: for any summation order |L~ - L| <= gamma ||x|| ||Wr_e||, gamma = 6 H 2^-24
//    (covers the tensor core's and the fixed-order fp32 path's roundings; Cauchy-Schwarz bounds
//    sum |x_h w_h|). The sigmoid is 1/4-Lipschitz, so every exact key lies in
//    [key~ - d_e, key~ + d_e], d_e = gamma ||x|| ||Wr_e|| / 4 + 2e-6 (the same sigmoid code on both
//    sides: its rounding and the bias addition are inside the 2e-6). With tau = the k-th largest
//    lower bound, an expert with upper bound < tau is below the k-th exact key: it cannot be
//    selected. Every other expert is a candidate.
// 3. router_exact_kernel: one warp per row recomputes the candidates' logits in the fixed chunked
//    order, then writes that row's keys (-inf for pruned experts) and scores for the top-k kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"
#include "router_math.cuh"

namespace moe {

constexpr int kScrRows = 128;        // rows (tokens) per CTA = MMA M
constexpr int kScrK = 64;            // bf16 elements of K per stage (128-byte rows)
constexpr int kScrStages = 4;
constexpr int kScrMaxE = 256;
constexpr int kCandMax = 64;
constexpr uint64_t kScrWaitNs = 1000000000ull;

bool router_screen_supported(const moe_shape* s) {
  return s->E <= kScrMaxE && s->H % kScrK == 0 && s->H <= 4096 && s->k <= s->E;
}

__global__ void router_norms_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, int T, int H,
                                    int E, float* __restrict__ xnorm, float* __restrict__ wnorm) {
  pdl_trigger();
  pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int r = warp; r < T + E; r += nwarps) {
    const uint16_t* row = r < T ? x + (size_t)r * H : wr + (size_t)(r - T) * H;
    float ss = 0.f;
    for (int h = lane * 8; h < H; h += 256) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + h));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = bf_lo(w[q]), b = bf_hi(w[q]);
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    // fp32 sum of squares is within H * 2^-24 (relative) of the exact value; 2^-10 covers it
    const float n = sqrtf(ss) * (1.0f + 0.0009765625f);
    if (lane == 0) {
      if (r < T) xnorm[r] = n;
      else wnorm[r - T] = n;
    }
  }
}

struct ScreenParams {
  const float* bias;
  const float* xnorm;
  const float* wnorm;
  int T, H, E, EP, k;
  float gamma4;          // gamma / 4
  int32_t* cand;         // [T, kCandMax]
  int32_t* ncand;        // [T]; -1 = too many candidates, recompute every expert
  uint32_t* status;
  const int32_t* anchor; // [T] or null: anchored rows need their own exact score of every expert
};

// Epilogue layout: 16 warps, four per TMEM lane quarter; warp group g (0..3) of a quarter takes
// the 16-column expert chunks g, g + 4, ... of the tile, so the 128 rows x E experts of bounds are
// computed by 512 threads. Each thread keeps the k largest lower bounds of its experts; one thread
// per row merges the four lists into tau (the k-th largest over all experts: the global top k is
// inside the union of the groups' top k).
constexpr int kScrEpiWarps = 16;
constexpr int kScrThreads = 128 + 32 * kScrEpiWarps;

static int screen_smem_bytes(int EP, int k) {
  const int stages = kScrStages * (kScrRows * kScrK * 2 + EP * kScrK * 2);
  const int scratch = EP * kScrRows * 4 + 4 * k * kScrRows * 4 + 2 * kScrRows * 4;
  return 1024 + 1024 + (stages > scratch ? stages : scratch);
}

__global__ void __launch_bounds__(kScrThreads, 1) router_screen_kernel(const __grid_constant__ CUtensorMap tmx,
                                                                        const __grid_constant__ CUtensorMap tmw,
                                                                        const ScreenParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // first 1 KB: barriers and flags; then the stage ring, reused after the mainloop as scratch
  uint64_t* full = reinterpret_cast<uint64_t*>(base);
  uint64_t* empty = full + kScrStages;
  uint64_t* accb = empty + kScrStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint8_t* ring = base + 1024;
  const int stageA = kScrRows * kScrK * 2;           // 16 KB
  const int stageB = p.EP * kScrK * 2;               // EP x 128 B
  const int stage_bytes = stageA + stageB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kScrRows;
  const int NS = p.H / kScrK;

  pdl_trigger();
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kScrStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    mbar_fence_init();
    prefetch_tmap(&tmx);
    prefetch_tmap(&tmw);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int s = 0; s < NS; ++s) {
        if (!mbar_wait(&empty[stage], phase ^ 1, kScrWaitNs, abort_flag, p.status, DEV_TIMEOUT_EMPTY)) break;
        uint8_t* sA = ring + stage * stage_bytes;
        mbar_arrive_expect_tx(&full[stage], stage_bytes);
        tma_load_2d(sA, &tmx, s * kScrK, t0, &full[stage]);
        tma_load_2d(sA + stageA, &tmw, s * kScrK, 0, &full[stage]);
        if (++stage == kScrStages) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16_f32(kScrRows, p.EP);
      for (int s = 0; s < NS; ++s) {
        if (!mbar_wait(&full[stage], phase, kScrWaitNs, abort_flag, p.status, DEV_TIMEOUT_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(ring + stage * stage_bytes), b0 = a0 + stageA;
#pragma unroll
        for (int kb = 0; kb < kScrK / 16; ++kb)
          mma_bf16(tmem, smem_desc(a0 + kb * 32, 16, 1024, 2), smem_desc(b0 + kb * 32, 16, 1024, 2), idesc,
                   (s > 0 || kb > 0) ? 1u : 0u);
        tc_commit(&empty[stage]);
        if (++stage == kScrStages) { stage = 0; phase ^= 1; }
      }
      // the accumulator barrier is committed on every path: after an expired wait this thread
      // itself waits on it (bounded, without the abort shortcut) so that no MMA it issued is still
      // running when TMEM is released
      tc_commit(accb);
      if (!ok) mbar_wait(accb, 0, kScrWaitNs, nullptr, nullptr, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int qd = warp & 3;                         // TMEM lane quarter
    const int g = (warp - 4) >> 2;                   // expert-chunk group
    const int tl = qd * 32 + lane;                   // row within the tile = TMEM lane
    const int tok = t0 + tl;
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    const int k = p.k;
    uint32_t okw = 1;
    if (lane == 0)
      okw = (mbar_wait(accb, 0, kScrWaitNs, abort_flag, p.status, DEV_TIMEOUT_ACCUM) && !*abort_flag) ? 1u : 0u;
    const bool ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
    tc_fence_after();
    // scratch (the stage ring is free now): lo[EP][128], lists[4][k][128], tau[128], count[128]
    float* lo = reinterpret_cast<float*>(ring);
    float* lists = lo + p.EP * kScrRows;
    float* tau_s = lists + 4 * k * kScrRows;
    int* cnt_s = reinterpret_cast<int*>(tau_s + kScrRows);
    const float xn = (tok < p.T) ? p.xnorm[tok] : 0.f;
    if (g == 0) cnt_s[tl] = 0;
    const int nch = p.EP / 16;
    if (ok) {
      for (int ch = g; ch < nch; ch += 4) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + ch * 16, r);
        tmem_ld_wait();
        reg_fence16(r);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int e = ch * 16 + c;
          if (e < p.E) {
            const float key = __fadd_rn(sigmoid_cw(__uint_as_float(r[c])), p.bias[e]);
            const float d = p.gamma4 * xn * p.wnorm[e] + 2e-6f;
            lo[e * kScrRows + tl] = key - d;
          }
        }
      }
      // this thread's k largest lower bounds (repeated maximum; taken entries set to -inf)
      for (int j = 0; j < k; ++j) {
        float best = -INFINITY;
        int be = -1;
        for (int ch = g; ch < nch; ch += 4)
          for (int c = 0; c < 16; ++c) {
            const int e = ch * 16 + c;
            if (e < p.E) {
              const float v = lo[e * kScrRows + tl];
              if (be < 0 || v > best) { best = v; be = e; }
            }
          }
        lists[(g * k + j) * kScrRows + tl] = best;
        if (be >= 0) lo[be * kScrRows + tl] = -INFINITY;
      }
    }
    named_bar_sync(1, 32 * kScrEpiWarps);
    if (ok && g == 0) {
      // tau = the k-th largest of the four lists
      float tau = -INFINITY;
      for (int j = 0; j < k; ++j) {
        float best = -INFINITY;
        int bi = 0;
        for (int i = 0; i < 4 * k; ++i) {
          const float v = lists[i * kScrRows + tl];
          if (v > best) { best = v; bi = i; }
        }
        tau = best;
        lists[bi * kScrRows + tl] = -INFINITY;
      }
      tau_s[tl] = tau;
    }
    named_bar_sync(1, 32 * kScrEpiWarps);
    // (the TMEM loads are warp-collective: every lane runs them; rows past T only skip the writes)
    if (ok) {
      const float tau = tau_s[tl];
      for (int ch = g; ch < nch; ch += 4) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + ch * 16, r);
        tmem_ld_wait();
        reg_fence16(r);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int e = ch * 16 + c;
          if (e < p.E && tok < p.T) {
            const float key = __fadd_rn(sigmoid_cw(__uint_as_float(r[c])), p.bias[e]);
            const float d = p.gamma4 * xn * p.wnorm[e] + 2e-6f;
            if (key + d >= tau) {
              const int n = atomicAdd(&cnt_s[tl], 1);
              if (n < kCandMax) p.cand[(size_t)tok * kCandMax + n] = e;
            }
          }
        }
      }
    }
    named_bar_sync(1, 32 * kScrEpiWarps);
    if (g == 0 && tok < p.T) {
      const int n = cnt_s[tl];
      // an anchored row is weighted by its own scores of its anchor's experts, which the screen
      // may have pruned: such rows recompute every expert exactly
      bool anchored = false;
      if (p.anchor) {
        const int a = p.anchor[tok];
        anchored = a >= 0 && a < p.T && p.anchor[a] == -1;
      }
      p.ncand[tok] = (!ok || n > kCandMax || anchored) ? -1 : n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// Exact recompute, one warp per CTA. The warp walks its rows t = blockIdx.x, + gridDim.x, ... as
// a stream of items: the row of x, then the Wr row of each candidate (every expert if the list
// overflowed). Items flow through a kExactStages-slot FIFO in shared memory, one TMA box per item
// (H/64 chunk rows of 128 bytes, 128-byte swizzle: the 16-byte unit j of chunk c sits at unit
// j ^ (c % 8), so the lanes' reads of chunks lane and lane + 32 fall in distinct banks). The row of
// x moves to registers when reached; a candidate item gives each lane the fixed-order partials of
// its two chunks (fp32 fused multiply-add of bf16 operands: one rounding per step, the same as
// widening first), and once per kExactBatch candidates (or at the row's end) lane b folds
// candidate b's partials in chunk order, applies the sigmoid and writes score and key. A row's keys
// are first written in full as -inf (scores 0), so pruned experts are never selected. The row
// metadata (count, candidate list) is loaded one row ahead of the producer. Waits are bounded; on
// expiry the kernel records DEV_TIMEOUT_FULL and stops.
constexpr int kExactBatch = 8;
constexpr int kExactStages = 4;

struct ExactItem {
  int t, j, e, cnt;                  // row, item index (-1 = x), expert, candidates in the row
};

// Slots start on 1024-byte boundaries: the 128-byte swizzle pattern is a function of the shared
// address, and the reads below assume it restarts at every slot.
__host__ __device__ inline int exact_slot_bytes(int NC) { return (NC * 128 + 1023) / 1024 * 1024; }

static size_t exact_smem_bytes(int H) {
  const int NC = H / kRouterChunk;
  return 1024 + (size_t)kExactStages * exact_slot_bytes(NC) + (size_t)kExactBatch * (NC + 1) * 4 + kExactBatch * 4 +
         kExactStages * (sizeof(ExactItem) + 8) + 16;
}

__global__ void __launch_bounds__(32, 16) router_exact_kernel(
    const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw, const float* __restrict__ bias,
    const int32_t* __restrict__ cand, const int32_t* __restrict__ ncand, int T, int H, int E,
    float* __restrict__ score, float* __restrict__ key, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t esm_raw[];
  uint8_t* esm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(esm_raw) + 1023) & ~uintptr_t(1023));
  const int NC = H / kRouterChunk;
  const int slot_bytes = exact_slot_bytes(NC);
  float* part = reinterpret_cast<float*>(esm + kExactStages * slot_bytes);   // [kExactBatch][NC + 1]
  int* re = reinterpret_cast<int*>(part + kExactBatch * (NC + 1));
  ExactItem* desc = reinterpret_cast<ExactItem*>(re + kExactBatch);
  uint64_t* full = reinterpret_cast<uint64_t*>(desc + kExactStages);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(full + kExactStages);
  const int lane = threadIdx.x;
  if (lane == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kExactStages; ++i) mbar_init(&full[i], 1);
    mbar_fence_init();
    prefetch_tmap(&tmx);
    prefetch_tmap(&tmw);
  }
  __syncwarp();
  pdl_trigger();
  pdl_wait();

  // ---- producer cursor (lane 0 issues): row p_t, item p_j; meta of this row and the next ----
  const int stride = gridDim.x;
  int p_t = blockIdx.x, p_j = -1;
  int p_nc = 0, p_cl0 = 0, p_cl1 = 0;
  int n_nc = 0, n_cl0 = 0, n_cl1 = 0;
  auto load_meta = [&](int t, int& nc, int& cl0, int& cl1) {
    if (t < T) {
      nc = ncand[t];
      cl0 = cand[(size_t)t * kCandMax + lane];
      cl1 = cand[(size_t)t * kCandMax + 32 + lane];
    }
  };
  load_meta(p_t, p_nc, p_cl0, p_cl1);
  load_meta(p_t + stride, n_nc, n_cl0, n_cl1);
  int ps = 0;
  auto produce = [&]() {
    ExactItem it{T, 0, 0, 0};
    if (p_t < T) {
      const int cnt = (p_nc < 0 || p_nc > kCandMax) ? E : p_nc;
      int e = 0;
      if (p_j >= 0) {
        const int v = __shfl_sync(0xffffffffu, p_j < 32 ? p_cl0 : p_cl1, p_j & 31);
        e = p_nc < 0 ? p_j : v;
      }
      if (lane == 0) {
        fence_async_smem();          // this slot's generic reads precede the copy that refills it
        mbar_arrive_expect_tx(&full[ps], (uint32_t)(NC * 128));
        if (p_j < 0) tma_load_2d(esm + ps * slot_bytes, &tmx, 0, p_t * NC, &full[ps]);
        else tma_load_2d(esm + ps * slot_bytes, &tmw, 0, e * NC, &full[ps]);
      }
      it = ExactItem{p_t, p_j, e, cnt};
      if (++p_j == cnt) {
        p_t += stride;
        p_j = -1;
        p_nc = n_nc;
        p_cl0 = n_cl0;
        p_cl1 = n_cl1;
        load_meta(p_t + stride, n_nc, n_cl0, n_cl1);
      }
    }
    if (lane == 0) desc[ps] = it;
    if (++ps == kExactStages) ps = 0;
  };

  for (int i = 0; i < kExactStages - 1; ++i) produce();
  uint32_t xr[2][32];                // the row's chunks lane and lane + 32 (bf16 pairs)
  int cs = 0, b = 0;
  uint32_t phase = 0;
  const int sw = (lane & 7) * 16;    // swizzle of chunks lane and lane + 32
  for (;;) {
    produce();
    __syncwarp();
    const ExactItem it = desc[cs];
    if (it.t >= T) break;
    uint32_t okw = 1;
    if (lane == 0) okw = mbar_wait(&full[cs], phase, kScrWaitNs, abort_flag, status, DEV_TIMEOUT_FULL) ? 1u : 0u;
    if (!__shfl_sync(0xffffffffu, okw, 0)) break;
    const uint8_t* slot = esm + cs * slot_bytes;
    if (it.j < 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = c < NC ? *reinterpret_cast<const uint4*>(slot + c * 128 + ((i * 16) ^ sw))
                                 : make_uint4(0, 0, 0, 0);
          xr[h][4 * i] = v.x;
          xr[h][4 * i + 1] = v.y;
          xr[h][4 * i + 2] = v.z;
          xr[h][4 * i + 3] = v.w;
        }
      }
      for (int e = lane; e < E; e += 32) {
        key[(size_t)it.t * E + e] = -INFINITY;
        score[(size_t)it.t * E + e] = 0.f;
      }
      b = 0;
    } else {
      // two independent 64-step chains (chunks lane and lane + 32), each in element order
      const uint8_t* w0 = slot + lane * 128;
      const uint8_t* w1 = slot + (lane + 32) * 128;
      const bool one = lane < NC, two = lane + 32 < NC;
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 a = one ? *reinterpret_cast<const uint4*>(w0 + ((i * 16) ^ sw)) : make_uint4(0, 0, 0, 0);
        const uint4 c = two ? *reinterpret_cast<const uint4*>(w1 + ((i * 16) ^ sw)) : make_uint4(0, 0, 0, 0);
        p0 = fma2_bf16(xr[0][4 * i], a.x, p0);
        p1 = fma2_bf16(xr[1][4 * i], c.x, p1);
        p0 = fma2_bf16(xr[0][4 * i + 1], a.y, p0);
        p1 = fma2_bf16(xr[1][4 * i + 1], c.y, p1);
        p0 = fma2_bf16(xr[0][4 * i + 2], a.z, p0);
        p1 = fma2_bf16(xr[1][4 * i + 2], c.z, p1);
        p0 = fma2_bf16(xr[0][4 * i + 3], a.w, p0);
        p1 = fma2_bf16(xr[1][4 * i + 3], c.w, p1);
      }
      if (one) part[b * (NC + 1) + lane] = p0;
      if (two) part[b * (NC + 1) + lane + 32] = p1;
      if (lane == 0) re[b] = it.e;
      ++b;
      if (b == kExactBatch || it.j + 1 == it.cnt) {
        __syncwarp();
        if (lane < b) {
          float acc = 0.f;
          for (int c = 0; c < NC; ++c) acc = __fadd_rn(acc, part[lane * (NC + 1) + c]);
          const int e = re[lane];
          const float sc = sigmoid_cw(acc);
          score[(size_t)it.t * E + e] = sc;
          key[(size_t)it.t * E + e] = __fadd_rn(sc, bias[e]);
        }
        b = 0;
      }
    }
    __syncwarp();
    if (++cs == kExactStages) {
      cs = 0;
      phase ^= 1;
    }
  }
  if (*abort_flag) {
    // copies still in flight land before the CTA's shared memory goes away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000) {
    }
  }
}

typedef CUresult (*EncodeTiledFnR)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static int make_bf16_tmap(CUtensorMap* m, const uint16_t* base, int cols, int rows, int box_rows) {
  static EncodeTiledFnR enc = nullptr;
  if (!enc) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return MOE_ERR_CUDA;
    enc = reinterpret_cast<EncodeTiledFnR>(ptr);
  }
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kScrK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), gdim, gstride, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

int launch_router_screen(const moe_shape* s, const uint16_t* x, const uint16_t* wr, const float* bias, void* ws,
                         float* score, float* key, cudaStream_t st, const int32_t* anchor) {
  const Workspace L = workspace_layout(s);
  const int T = s->T, H = s->H, E = s->E;
  float* xnorm = ws_ptr<float>(ws, L.xnorm);
  float* wnorm = ws_ptr<float>(ws, L.wnorm);
  int32_t* cand = ws_ptr<int32_t>(ws, L.cand);
  int32_t* ncand = ws_ptr<int32_t>(ws, L.ncand);
  const int nb = (int)std::min<long long>(((long long)(T + E) * 32 + 255) / 256, (long long)num_sms() * 8);
  int rc = launch_pdl(router_norms_kernel, dim3(nb), dim3(256), 0, st, x, wr, T, H, E, xnorm, wnorm);
  if (rc) return rc;
  ScreenParams sp{};
  sp.bias = bias;
  sp.xnorm = xnorm;
  sp.wnorm = wnorm;
  sp.T = T;
  sp.H = H;
  sp.E = E;
  sp.EP = (E + 15) / 16 * 16;
  sp.k = s->k;
  sp.gamma4 = (float)(6.0 * H / 16777216.0 / 4.0);
  sp.cand = cand;
  sp.ncand = ncand;
  sp.status = ws_ptr<uint32_t>(ws, L.status);
  sp.anchor = anchor;
  CUtensorMap tmx, tmw;
  rc = make_bf16_tmap(&tmx, x, H, T, kScrRows);
  if (rc) return rc;
  rc = make_bf16_tmap(&tmw, wr, H, E, sp.EP);
  if (rc) return rc;
  const int smem = screen_smem_bytes(sp.EP, sp.k);
  if (ensure_smem_limit((const void*)router_screen_kernel, smem)) return MOE_ERR_CUDA;
  rc = launch_pdl(router_screen_kernel, dim3(ceil_div(T, kScrRows)), dim3(kScrThreads), (size_t)smem, st, tmx, tmw,
                  sp);
  if (rc) return rc;
  CUtensorMap tex, tew;
  const int NC = H / kRouterChunk;
  rc = make_bf16_tmap(&tex, x, kRouterChunk, T * NC, NC);
  if (rc) return rc;
  rc = make_bf16_tmap(&tew, wr, kRouterChunk, E * NC, NC);
  if (rc) return rc;
  const size_t esmem = exact_smem_bytes(H);
  if (ensure_smem_limit((const void*)router_exact_kernel, (int)esmem)) return MOE_ERR_CUDA;
  const int eper_sm = ctas_per_sm_by_smem(esmem, 16);
  const int eg = (int)std::min<long long>(T, (long long)num_sms() * eper_sm);
  return launch_pdl(router_exact_kernel, dim3(eg), dim3(32), esmem, st, tex, tew, bias, cand, ncand, T, H, E, score,
                    key, sp.status);
}

}  // namespace moe
