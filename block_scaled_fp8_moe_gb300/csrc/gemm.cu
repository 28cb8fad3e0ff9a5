// Grouped block-scaled GEMMs of the routed experts on tcgen05 (sm_103a).
//
// "New Deepseek 4.1 flash recipe", post 6 "How it works" items 1-2: routed experts run FP8
// activations x FP4 weights through a block-scaled MMA (kind::mxf8f6f4); decode rows run on
// 16/32/64-row tiles; prefill rasterises weights larger than L2 in panels. Post 4 "Fenced
// pipeline stages": a stage may be refilled only after every read of it has completed.
// TP4 serving profile README, "Experts" row: per-slot output buffer, fixed-order sum.
//
// Shape of one CTA work item: 128 weight rows (MMA M) x BN plan rows (MMA N, tokens), K looped in
// 128-element chunks. Weights sit on the A side so decode and prefill share one accumulation
// order for every output element: the K loop is identical, never split, and a token's column
// position does not change the arithmetic of its column.
//
// Roles (256 threads; 384 for 128-row token tiles):
//   warp 0      TMA producer: packed weight tile (FP4, unpacked to 8-bit containers by the TMA)
//               and its 512-byte scale block (bulk copy); one mbarrier transaction per stage.
//   warps 1, 3  token-operand producers: cp.async gathers of the BN activation rows (128 B each,
//               128B-swizzled in shared memory) and their scale bytes for narrow tiles; for wide
//               tiles warp 1 loads one TMA box of plan-order rows per K-chunk and writes the scale
//               atoms with 16-byte shared stores. Both arrive on the same stage mbarrier.
//   warp 2      TMEM owner and MMA issuer: tcgen05.cp of the scale blocks to TMEM, four K=32
//               MMAs per K-chunk, tcgen05.commit releases the stage only after the MMAs (and
//               copies) that read it are complete.
//   warps 4-7   epilogue (and 8-11 for 128-row tiles): tcgen05.ld of the fp32 accumulator, SwiGLU +
//               MXFP8 requant (W13) or routing-weight scaling into the per-slot buffer (W2).
// Work items (expert, weight panel, token tile) are walked with the token tile fastest, so CTAs
// running at the same time share one weight panel through L2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "combine.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "mx.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {

#ifndef MOE_KT_WIDE
#define MOE_KT_WIDE 2               // K-chunks per stage for 128-row token tiles
#endif
#ifndef MOE_WIDE_BN
#define MOE_WIDE_BN 224             // widest token tile (MMA N) of the prefill path
#endif
#ifndef MOE_WIDE_STAGES
#define MOE_WIDE_STAGES 2           // pipeline stages of the widest tiles
#endif
#ifndef MOE_WIDE_KT
#define MOE_WIDE_KT 1               // K-chunks per stage of the widest tiles
#endif
#ifndef MOE_PANEL_FAST
#define MOE_PANEL_FAST 0            // 1: work items walk the weight panels fastest (token tile outer)
#endif
#ifndef MOE_N128_CTAS
#define MOE_N128_CTAS 1             // CTAs per SM of 128-row token tiles (2: one accumulator each)
#endif
#ifndef MOE_WIDE_CTAS
#define MOE_WIDE_CTAS 2             // CTAs per SM of the widest tiles (2: one accumulator each)
#endif
// 4 producer/MMA warps + 4 epilogue warps; 128-row token tiles (one CTA per SM) take 8 epilogue
// warps (two per TMEM lane quarter, splitting the tile's columns), since their epilogue, not the
// MMA, sets the pace. The widest tiles run two CTAs per SM with 4 epilogue warps each.
template <int BN>
struct Threads {
  static constexpr int kEpiWarps = ((BN == 128 && MOE_N128_CTAS == 1) || (BN > 128 && MOE_WIDE_CTAS == 1)) ? 8 : 4;
  static constexpr int kCount = 128 + 32 * kEpiWarps;
};
#ifndef MOE_DEC_KT
#define MOE_DEC_KT 1                // K-chunks per stage, decode tiles (16 / 32 token rows)
#endif
#ifndef MOE_DEC_STAGES
#define MOE_DEC_STAGES 2
#endif
#ifndef MOE_DEC_CTAS
#define MOE_DEC_CTAS 4              // decode-tile CTAs per SM
#endif
#ifndef MOE_DEC_PF
#define MOE_DEC_PF 2                // weight tiles prefetched into L2 ahead of the loads, decode tiles
#endif
#ifndef MOE_WIDE_PF
#define MOE_WIDE_PF 0               // the same for 64-row and wider token tiles
#endif

__host__ __device__ constexpr int pow2_at_least(int v, int p) { return p >= v ? p : pow2_at_least(v, 2 * p); }

template <int BN>
struct Smem {
  // A pipeline stage holds KT consecutive K-chunks (weight tiles) of 128. A CTA completes a stage
  // in a roughly fixed time, so the bytes per stage and the CTAs per SM set its streaming rate:
  // decode tiles run 4 CTAs/SM of 2 one-chunk stages, 128-row tiles stages of two chunks.
  static constexpr int KT =
      (BN <= 32) ? MOE_DEC_KT : (BN <= 64 ? 1 : (BN == 128 ? (MOE_N128_CTAS == 2 ? 1 : MOE_KT_WIDE) : MOE_WIDE_KT));
  static constexpr int kTileA = 16384;                           // one unpacked 128 x 128 FP4 tile
  static constexpr int kTileB = BN * 128;                        // BN rows x 128 FP8
  static constexpr int kStageA = KT * kTileA;
  static constexpr int kStageB = KT * kTileB;
  static constexpr int kSfbChunk = 512 * ((BN + 127) / 128);     // B scale atoms of one K-chunk
  static constexpr int kSfChunk = 512 + kSfbChunk;
  static constexpr int kStageBytes = (int)((kStageA + kStageB + KT * kSfChunk + 1023) / 1024 * 1024);
  static constexpr int kStages =
      (BN <= 32) ? MOE_DEC_STAGES
                 : (BN <= 64 ? 3 : (BN == 128 ? (MOE_N128_CTAS == 2 ? 2 : 6 / MOE_KT_WIDE) : MOE_WIDE_STAGES));
  static constexpr int kCtasPerSm =
      (BN <= 32) ? MOE_DEC_CTAS : (BN <= 64 ? 2 : (BN == 128 ? MOE_N128_CTAS : MOE_WIDE_CTAS));
  // accumulator slots in TMEM: two (the epilogue of one tile overlaps the next tile's MMAs), or
  // one when two wide CTAs share the SM (the other CTA's MMAs fill the epilogue's time)
  static constexpr int kAcc = ((BN == 128 && MOE_N128_CTAS == 2) || (BN > 128 && MOE_WIDE_CTAS == 2)) ? 1 : 2;
  // the weight producer keeps kPrefetch K-chunks of its own upcoming tiles (codes and scales)
  // requested into L2 beyond the stages in flight: more bytes in flight per SM than shared memory
  // holds, so a stage's load finds its data in L2 instead of waiting a full DRAM round trip
  static constexpr int kPrefetch = (BN <= 32) ? MOE_DEC_PF : MOE_WIDE_PF;
  // TMEM: kAcc accumulator slots of kAccStride columns, then the ring of scale blocks (one slot of
  // kSfSlot columns per K-chunk in flight: 4 for A, 4 per 128 token rows for B); the allocation is
  // the next power of two, small enough for kCtasPerSm CTAs to share the SM's 512 columns
  static constexpr int kAccStride = (BN <= 32) ? 32 : (BN <= 64 ? 64 : BN);
  static constexpr int kSfCol = kAcc * kAccStride;
  static constexpr int kSfSlot = 4 + 4 * ((BN + 127) / 128);
  static constexpr int kTmemCols = pow2_at_least(kSfCol + kStages * KT * kSfSlot, 32);
  static_assert(kTmemCols * kCtasPerSm <= 512, "TMEM columns per SM");
  static_assert(kSfCol + kStages * KT * kSfSlot <= kTmemCols, "TMEM columns");
  // wide token tiles read the activation operand with TMA (one 2D box of plan-order rows per
  // K-chunk) instead of cp.async gathers, and size each expert's tiles to its row count
  static constexpr bool kTmaB = (BN >= 128);
  static constexpr int kTiles = kStages * kStageBytes;
  static constexpr int kXchg = 2 * 64 * 16 * 4 * (Threads<BN>::kEpiWarps / 4);   // W13 epilogue exchange
  static constexpr int kMisc = 1024;                            // barriers, flags
  static constexpr int kRows = 128 * 8;                         // gather row table
  static constexpr int kFixed = 1024 + kTiles + kXchg + kMisc + kRows;
  // + plan tables sized per launch: (E + 1) x (offsets, tile starts) ints, and a second table of
  // tile starts when one launch runs both GEMMs; + when the launch plans for itself, a token bitmask
  // per expert and per slot its expert, weight, plan row and (indexed by plan row) its slot
  static int total(int E, bool two_gemms, int self_plan_slots = 0) {
    return kFixed + (int)align_up((size_t)(E + 1) * (two_gemms ? 12 : 8), 16) +
           (self_plan_slots ? (int)align_up((size_t)E * 4 + (size_t)self_plan_slots * 16, 16) : 0);
  }
  static_assert(kFixed + (kMaxE + 1) * 8 + 16 <= 227 * 1024, "shared memory per CTA at the largest E");
};

// MODE 0: the down projection (W2); 1: gate/up with SwiGLU and requant (W13); 2: W13 then W2 in
// one persistent launch (decode tiles): every CTA works through its W13 items, then its W2 items;
// 3: mode 2 for a batch of at most kSelfPlanMaxT rows that routes itself: every CTA takes the top-k
// of the rows from the router's scores (a warp per row, the plan kernel's selection) and builds
// the plan in its shared memory, so no plan kernel runs between the router and the GEMMs.
// A W2 item's weight tiles stream as soon as the CTA reaches it; its token rows (h) are gathered
// once the W13 epilogues have counted every W13 tile of that expert (GemmParams::ready). All CTAs
// are resident (the grid is sized to the GPU), and each CTA finishes its W13 items before its W2
// ones, so every counted tile is produced by a CTA that is running. In mode 2, p describes W13 and
// p2 / tmap_a2 the down projection; otherwise p2 and tmap_a2 repeat p and tmap_a.
template <int BN, int MODE>
__global__ void __launch_bounds__(Threads<BN>::kCount, Smem<BN>::kCtasPerSm)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_a2, const __grid_constant__ GemmParams p,
                        const __grid_constant__ GemmParams p2) {
  using L = Smem<BN>;
  constexpr bool kFused = MODE >= 2;
  constexpr bool kSelfPlan = MODE == 3;
  constexpr bool kW13Only = MODE == 1;
  constexpr int S = L::kStages;
  constexpr int NACC = L::kAcc;                    // accumulator slots in TMEM
  constexpr bool kTmaB = L::kTmaB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = base;
  float* xchg = reinterpret_cast<float*>(base + L::kTiles);
  uint8_t* misc = base + L::kTiles + L::kXchg;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;          // [NACC]
  uint64_t* acc_empty = acc_full + 2;      // [NACC]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  long long* s_rows = reinterpret_cast<long long*>(misc + L::kMisc);   // [BN] gather row or -1
  int* s_off = reinterpret_cast<int*>(misc + L::kMisc + L::kRows);      // expert offsets [E+1]
  int* s_cum = s_off + (p.E + 1);                                       // MT * tile starts [E+1]
  int* s_cum2 = s_cum + (p.E + 1);                                      // the same for p2.MT (mode 2)
  // mode 3: the plan built here (nsl = T k slots)
  const int nsl = kSelfPlan ? p.T * p.k : 0;
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_cum2 + (p.E + 1));   // live rows choosing e, bit t
  int* s_se = reinterpret_cast<int*>(s_mask + p.E);                     // slot -> expert
  float* s_sw = reinterpret_cast<float*>(s_se + nsl);                   // slot -> routing weight
  int* s_ros = s_se + 2 * nsl;                                          // slot -> plan row or -1
  int* s_sor = s_se + 3 * nsl;                                          // plan row -> slot

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;

  // ---- prologue: barriers and TMEM (overlaps the previous kernel), then the plan tables ----
  pdl_trigger();
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + (kTmaB ? 32 : 64));
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], Threads<BN>::kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_a);
    if (kTmaB) prefetch_tmap(&tmap_b);
  }
  if (kSelfPlan) {
    for (int i = threadIdx.x; i < E; i += Threads<BN>::kCount) s_mask[i] = 0;
    __syncthreads();
  }
  pdl_wait();                                    // everything below may read upstream results
  if (kSelfPlan) {
    // top-k of row t on warp t % 8, rows in turn (the choices and weights of the plan kernel); a live
    // row sets its bit in the masks of its k experts
    for (int t = warp; t < p.T; t += Threads<BN>::kCount / 32) {
      int my_e = 0;
      float my_s = 0.f, sum = 0.f;
      const float2* srow = p.sel + ((size_t)(blockIdx.x % kSelfPlanReplicas) * p.T + t) * E;
      warp_topk<kSelfPlanNI, true>(reinterpret_cast<const float*>(srow), nullptr, E, p.k, lane, nullptr, &my_e,
                                   &my_s, &sum);
      const bool live = p.dead == nullptr || p.dead[t] == 0;
      if (lane < p.k) {
        s_se[t * p.k + lane] = my_e;
        s_sw[t * p.k + lane] = __fdiv_rn(my_s, sum);
        if (live) atomicOr(&s_mask[my_e], 1u << t);
      }
    }
    __syncthreads();
    if (warp == 0) {
      // offsets and tile starts: warp-parallel prefix sums of count_e and ceil(count_e / BN); lane l
      // takes experts l per .. l per + per - 1 (per <= kSelfPlanNI), all its mask loads in flight
      const int per = (E + 31) / 32;
      const int e0 = lane * per;
      int cnt[kSelfPlanNI];
      int lc = 0, lt = 0;
#pragma unroll
      for (int j = 0; j < kSelfPlanNI; ++j) {
        const int e = e0 + j;
        cnt[j] = (j < per && e < E) ? __popc(s_mask[e]) : 0;
        lc += cnt[j];
        lt += (cnt[j] + BN - 1) / BN;
      }
      int ic = lc, it = lt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int vc = __shfl_up_sync(0xffffffffu, ic, off);
        const int vt = __shfl_up_sync(0xffffffffu, it, off);
        if (lane >= off) {
          ic += vc;
          it += vt;
        }
      }
      int rc = ic - lc, rt = it - lt;
      const int mt1 = p.MT, mt2 = p2.MT;
#pragma unroll
      for (int j = 0; j < kSelfPlanNI; ++j) {
        const int e = e0 + j;
        if (j < per && e < E) {
          s_off[e] = rc;
          s_cum[e] = rt * mt1;
          s_cum2[e] = rt * mt2;
        }
        rc += cnt[j];
        rt += (cnt[j] + BN - 1) / BN;
      }
      if (lane == 31) {
        s_off[E] = ic;
        s_cum[E] = it * p.MT;
        s_cum2[E] = it * p2.MT;
      }
      __syncwarp();
      // a live slot's plan row: its expert's offset plus the expert's rows of lower tokens
#pragma unroll 2
      for (int i = lane; i < nsl; i += 32) {
        const int t = i / p.k;
        const int e = s_se[i];
        const uint32_t bits = s_mask[e];
        int row = -1;
        if ((bits >> t) & 1u) {
          row = s_off[e] + __popc(bits & ((1u << t) - 1u));
          s_sor[row] = i;
        }
        s_ros[i] = row;
      }
    }
  } else {
    for (int i = threadIdx.x; i <= E; i += Threads<BN>::kCount) s_off[i] = p.offsets[i];
    __syncthreads();
    if (warp == 0) {
      // tile starts: warp-parallel prefix sum of ceil(count_e / BN), times MT
      const int per = (E + 31) / 32;
      const int e0 = lane * per;
      int local = 0;
      for (int e = e0; e < min(E, e0 + per); ++e) local += (s_off[e + 1] - s_off[e] + BN - 1) / BN;
      int incl = local;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      int run = incl - local;
      for (int e = e0; e < min(E, e0 + per); ++e) {
        s_cum[e] = run * p.MT;
        if (kFused) s_cum2[e] = run * p2.MT;
        run += (s_off[e + 1] - s_off[e] + BN - 1) / BN;
      }
      if (lane == 31) {
        s_cum[E] = incl * p.MT;
        if (kFused) s_cum2[E] = incl * p2.MT;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total1 = s_cum[E];                        // items of the first (or only) GEMM
  const int total = total1 + (kFused ? s_cum2[E] : 0);

  // decode work item w -> (GEMM, e, m, nt); first = the item belongs to p (W13 in mode 2); tw = the
  // expert's tile width (columns per token tile): BN for narrow tiles, else its rows spread evenly
  // over ceil(count / BN) tiles, rounded up to 16
  auto decode = [&](int w, bool& first, int& e, int& m, int& nt, int& row0, int& nrows, int& tw) {
    first = !kFused || w < total1;
    const int* cum = first ? s_cum : s_cum2;
    const int MT = first ? p.MT : p2.MT;
    const int ww = first ? w : w - total1;
    e = find_expert(cum, E, ww);
    const int cnt = s_off[e + 1] - s_off[e];
    const int ntiles = (cnt + BN - 1) / BN;
    tw = BN;
    if (kTmaB) tw = min(BN, ((cnt + ntiles - 1) / ntiles + 15) / 16 * 16);
    const int local = ww - cum[e];
    if (MOE_PANEL_FAST) {
      nt = local / MT;
      m = local - nt * MT;
    } else {
      m = local / ntiles;
      nt = local - m * ntiles;
    }
    row0 = s_off[e] + nt * tw;
    nrows = min(tw, cnt - nt * tw);
  };
  // the gate/up GEMM (SwiGLU epilogue) or the down projection, for an item of GEMM `first`
  auto is_w13 = [&](bool first) { return kFused ? first : kW13Only; };

  if (warp == 0) {
    // ===================== TMA producer: weights =====================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t tile_bytes = p.a_fp8 ? 2 * kTileCodeBytes : kTileCodeBytes;
      // L2 prefetch cursor: walks this CTA's (item, K-chunk) sequence kPrefetch chunks ahead of
      // the loads. It starts kPrefetch chunks in without prefetching: the first chunks are loaded
      // at once, and a burst of prefetches for them would only queue ahead of those loads.
      int pf_w = blockIdx.x, pf_kc = 0;
      long long pf_tile0 = -1;
      auto pf_step = [&](bool issue) {
        if (pf_w >= total) return;
        const bool pf_first = !kFused || pf_w < total1;
        const GemmParams& pq = pf_first ? p : p2;
        if (issue) {
          if (pf_tile0 < 0) {
            int e, m, nt, row0, nrows, tw;
            bool first;
            decode(pf_w, first, e, m, nt, row0, nrows, tw);
            pf_tile0 = (long long)(e * pq.MT + m) * pq.KC;
          }
          const long long g = pf_tile0 + pf_kc;
          prefetch_l2_bulk(pq.a_codes + g * tile_bytes, tile_bytes);
          prefetch_l2_bulk(pq.a_scales + g * kTileScaleBytes, kTileScaleBytes);
        }
        if (++pf_kc == pq.KC) {
          pf_kc = 0;
          pf_w += gridDim.x;
          pf_tile0 = -1;
        }
      };
      for (int i = 0; i < L::kPrefetch; ++i) pf_step(false);
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        int e, m, nt, row0, nrows, tw;
        bool first;
        decode(w, first, e, m, nt, row0, nrows, tw);
        const GemmParams& q = first ? p : p2;
        const CUtensorMap* ta = first ? &tmap_a : &tmap_a2;
        const int KC = q.KC;
        const int tile0 = (e * q.MT + m) * KC;
        for (int kc0 = 0; kc0 < KC; kc0 += L::KT) {
          if (!mbar_wait(&empty[stage], phase ^ 1, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_EMPTY)) {
            ok = false;
            break;
          }
          const int nv = min(L::KT, KC - kc0);            // chunks of this stage inside the panel
          uint8_t* sA = tiles + stage * L::kStageBytes;
          uint8_t* sSFA = sA + L::kStageA + L::kStageB;
          // the box always moves KT tiles (past the panel: the next panel's tiles or TMA fill);
          // the scale copy stops at the panel's end
          mbar_arrive_expect_tx(&full[stage], L::KT * (p.a_fp8 ? 2 * kTileCodeBytes : kTileCodeBytes) + nv * kTileScaleBytes +
                                                  (kTmaB ? L::kStageB : 0));
          tma_load_2d(sA, ta, 0, (tile0 + kc0) * 128, &full[stage]);
          bulk_load(sSFA, q.a_scales + (size_t)(tile0 + kc0) * kTileScaleBytes, nv * kTileScaleBytes, &full[stage]);
          if (L::kPrefetch > 0)
            for (int j = 0; j < nv; ++j) pf_step(true);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
    } else if (kSelfPlan && blockIdx.x == 0) {
      // the plan, for the caller: written by CTA 0 on this warp's otherwise idle lanes 1..31
      for (int i = lane - 1; i < nsl; i += 31) {
        p.plan_topk_idx[i] = s_se[i];
        p.plan_topk_w[i] = s_sw[i];
        p.plan_row_of_slot[i] = s_ros[i];
        if (s_ros[i] >= 0) p.plan_slot_of_row[s_ros[i]] = i;
      }
      for (int e = lane - 1; e <= E; e += 31) {
        p.plan_offsets[e] = s_off[e];
        if (e < E) p.plan_counts[e] = __popc(s_mask[e]);
      }
    }
  } else if (kTmaB && warp == 1) {
    // ===================== TMA producer: activations (wide token tiles) =====================
    // The token operand of a wide tile is always in plan order (W2: hq; W13: a copy of xq gathered
    // into plan order before the GEMM), so lane 0 loads the tile's contiguous plan rows with one
    // 2D TMA box; rows past the tile's end belong to the next expert (or are TMA zero fill) and
    // their columns are never stored. The lanes also write the stage's scale atoms with 16-byte
    // shared stores, make them visible to the MMA's async proxy and arrive on the stage barrier.
    // Stages stream in order (items w, K-chunk groups kc0); a stage's scale words are loaded one
    // stage ahead, before the previous stage's are stored, so their latency overlaps a whole stage.
    constexpr int NA = (BN + 127) / 128;
    int w = blockIdx.x, kn = 0;
    int e = 0, m = 0, nt = 0, row0 = 0, nrows = 0, tw = 0;
    bool first = true;
    if (w < total) decode(w, first, e, m, nt, row0, nrows, tw);
    auto next_stage = [&](int& r0, int& nr, int& kc0) {        // the stage at the cursor, then advance
      if (w >= total) return false;
      r0 = row0;
      nr = nrows;
      kc0 = kn;
      kn += L::KT;
      if (kn >= p.KC) {
        kn = 0;
        w += gridDim.x;
        if (w < total) decode(w, first, e, m, nt, row0, nrows, tw);
      }
      return true;
    };
    auto load_stage = [&](ScaleLines<NA>(&sl)[L::KT], int r0, int nr, int kc0) {
#pragma unroll
      for (int j = 0; j < L::KT; ++j)
        if (kc0 + j < p.KC) load_scale_lines<NA>(sl[j], p.bs, p.b_scale_pitch, r0, nr, kc0 + j, lane);
    };
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int r0 = 0, nr = 0, kc0 = 0;
    bool have = next_stage(r0, nr, kc0);
    ScaleLines<NA> sl[L::KT];
    if (have) load_stage(sl, r0, nr, kc0);
    while (have) {
      int r1 = 0, nr1 = 0, kc1 = 0;
      const bool have1 = next_stage(r1, nr1, kc1);
      ScaleLines<NA> sl1[L::KT];
      if (have1) load_stage(sl1, r1, nr1, kc1);
      if (ok) ok = warp_wait(&empty[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_EMPTY);
      if (ok) {
        uint8_t* sB0 = tiles + stage * L::kStageBytes + L::kStageA;
        uint8_t* sSFB0 = sB0 + L::kStageB + L::KT * 512;
        // every stage moves KT boxes of BN rows (the transaction count the weight producer
        // announced); rows past the tile and boxes past the end of K are never multiplied
        if (lane == 0)
          for (int j = 0; j < L::KT; ++j)
            tma_load_2d(sB0 + j * L::kTileB, &tmap_b, (kc0 + j) * 128, r0, &full[stage]);
#pragma unroll
        for (int j = 0; j < L::KT; ++j)
          if (kc0 + j < p.KC) store_scale_lines<NA>(sl[j], sSFB0 + j * L::kSfbChunk, lane);
        fence_async_smem();
        mbar_arrive(&full[stage]);
      }
      if (++stage == S) { stage = 0; phase ^= 1; }
      have = have1;
      r0 = r1;
      nr = nr1;
      kc0 = kc1;
#pragma unroll
      for (int j = 0; j < L::KT; ++j) sl[j] = sl1[j];
    }
  } else if (!kTmaB && (warp == 1 || warp == 3)) {
    // ===================== gather producers: activations =====================
    // After an expired wait the loops keep running (doing nothing) so that both warps meet at
    // every named barrier.
    const int pb = (warp == 1 ? 0 : 32) + lane;       // 0..63
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
      int e, m, nt, row0, nrows, tw;
      bool first;
      decode(w, first, e, m, nt, row0, nrows, tw);
      const GemmParams& q = first ? p : p2;
      named_bar_sync(2, 64);                          // previous item's table no longer in use
      for (int c = pb; c < BN; c += 64) {
        long long r = -1;
        if (c < nrows) {
          const int prow = row0 + c;
          r = (is_w13(first) && !q.b_plan_rows)
                  ? (long long)((kSelfPlan ? s_sor[prow] : q.slot_of_row[prow]) / q.k)
                  : (long long)prow;
        }
        s_rows[c] = r;
      }
      named_bar_sync(2, 64);
      if (kFused && !first && ok) {
        // the expert's h rows exist once every W13 tile of the expert has been counted
        const uint32_t need = (uint32_t)((s_cum[e + 1] - s_cum[e]) * Threads<BN>::kEpiWarps);
        uint32_t got = 1;
        if (lane == 0) got = wait_count_at_least(q.ready + e, need, kWaitLimitNs, abort_flag, q.status) ? 1u : 0u;
        ok = __shfl_sync(0xffffffffu, got, 0) != 0;
        __syncwarp();                                 // the lanes' gathers follow lane 0's acquire
      }
      for (int kc0 = 0; kc0 < q.KC; kc0 += L::KT) {
        if (ok) ok = warp_wait(&empty[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_EMPTY);
        if (ok) {
          const int nv = min(L::KT, q.KC - kc0);
          uint8_t* sB0 = tiles + stage * L::kStageBytes + L::kStageA;
          uint8_t* sSFB0 = sB0 + L::kStageB + L::KT * 512;
          for (int j2 = 0; j2 < nv; ++j2) {
            const int kc = kc0 + j2;
            uint8_t* sB = sB0 + j2 * L::kTileB;
            uint8_t* sSFB = sSFB0 + j2 * L::kSfbChunk;
            for (int i = pb; i < BN * 8; i += 64) {
              const int c = i >> 3, j = i & 7;
              const long long r = s_rows[c];
              const int kbyte = kc * 128 + j * 16;
              const bool valid = (r >= 0) && (kbyte < q.b_row_bytes);
              const uint8_t* src = valid ? q.bq + r * q.b_row_bytes + kbyte : q.bq;
              cp_async_16(sB + c * 128 + ((j ^ (c & 7)) << 4), src, valid ? 16u : 0u);
            }
            for (int c = pb; c < BN; c += 64) {
              const long long r = s_rows[c];
              const bool valid = r >= 0;
              const uint8_t* src = valid ? q.bs + r * q.b_scale_pitch + kc * 4 : q.bs;
              cp_async_4(sSFB + (c & 31) * 16 + (c >> 5) * 4, src, valid ? 4u : 0u);
            }
          }
          cp_async_arrive_noinc(&full[stage]);
        }
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
    cp_async_wait_all();
  } else if (warp == 2) {
    // ===================== MMA issuer =====================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++it) {
        int e, m, nt, row0, nrows, tw;
        bool first;
        decode(w, first, e, m, nt, row0, nrows, tw);
        const GemmParams& q = first ? p : p2;
        const uint32_t idesc_base = idesc_mxf8f6f4(p.a_fp8 ? 0 : 5 /*weights E4M3 or E2M1*/, 0 /*E4M3*/, 128, tw, 0, 0);
        const int acc = (NACC == 2) ? (it & 1) : 0;
        const int use = (NACC == 2) ? (it >> 1) : it;       // how many times this slot was used before
        if (use > 0 &&
            !mbar_wait(&acc_empty[acc], (use - 1) & 1, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_DRAIN)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * L::kAccStride);
        for (int kc0 = 0; kc0 < q.KC; kc0 += L::KT) {
          if (!mbar_wait(&full[stage], phase, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_FULL)) {
            ok = false;
            break;
          }
          // narrow tiles' token rows and scales arrive by cp.async (generic proxy): make them visible
          // to the MMA's async proxy here; the wide tiles' producer fences its own stores before it
          // arrives on the stage barrier
          if (!kTmaB) fence_async_smem();
          tc_fence_after();
          const int nv = min(L::KT, q.KC - kc0);
          uint8_t* sA0 = tiles + stage * L::kStageBytes;
          uint8_t* sB0 = sA0 + L::kStageA;
          uint8_t* sSFA0 = sB0 + L::kStageB;
          uint8_t* sSFB0 = sSFA0 + L::KT * 512;
          for (int j = 0; j < nv; ++j) {
            const int kc = kc0 + j;
            const uint32_t tsfa = tmem + L::kSfCol + (stage * L::KT + j) * L::kSfSlot;
            const uint32_t tsfb = tsfa + 4;
            tc_cp_32x128b_warpx4(tsfa, smem_desc(smem_u32(sSFA0 + j * 512), 16, 128, 0));
            // B scales: one 512-byte atom per 128 token rows, atom q at TMEM column tsfb + 4 q
            for (int a = 0; a * 128 < tw; ++a)
              tc_cp_32x128b_warpx4(tsfb + 4 * a, smem_desc(smem_u32(sSFB0 + j * L::kSfbChunk + a * 512), 16, 128, 0));
            const uint32_t a0 = smem_u32(sA0 + j * L::kTileA), b0 = smem_u32(sB0 + j * L::kTileB);
            const int nk = min(4, (q.K - kc * 128) / 32);
            for (int kb = 0; kb < nk; ++kb) {
              const uint64_t ad = smem_desc(a0 + kb * 32, 16, 1024, 2);
              const uint64_t bd = smem_desc(b0 + kb * 32, 16, 1024, 2);
              const uint32_t id = idesc_base | ((uint32_t)kb << 4) | ((uint32_t)kb << 29);
              mma_mxf8f6f4(d_tmem, ad, bd, id, tsfa, tsfb, (kc > 0 || kb > 0) ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
      }
      // every MMA and scale copy this thread issued has completed before TMEM is released: the
      // commit arrives once they finish, also after an abort, so this wait does not take the
      // abort shortcut (it stays bounded by its own limit)
      tc_commit(drain);
      mbar_wait(drain, 0, kWaitLimitNs, nullptr, p.status, DEV_TIMEOUT_DRAIN);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ===================== epilogue (warp w -> TMEM lanes 32 (w % 4)) =====================
    // With 8 epilogue warps, warps 4-7 take the even column groups of a tile and warps 8-11 the
    // odd ones, each set with its own exchange buffer and named barrier. As above, an expired wait
    // turns the remaining iterations into no-ops that still meet at the named barriers.
    constexpr int kHalves = Threads<BN>::kEpiWarps / 4;
    const int qd = (warp - 4) & 3;                    // TMEM lane quarter of this warp
    const int half = (warp - 4) >> 2;
    const uint32_t bar_id = 1 + 2 * half;
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    int it = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++it) {
      int e, m, nt, row0, nrows, tw;
      bool first;
      decode(w, first, e, m, nt, row0, nrows, tw);
      const GemmParams& q = first ? p : p2;
      const bool w13_item = is_w13(first);
      const int acc = (NACC == 2) ? (it & 1) : 0;
      const int use = (NACC == 2) ? (it >> 1) : it;
      if (ok) ok = warp_wait(&acc_full[acc], use & 1, abort_flag, p.status, DEV_TIMEOUT_ACCUM);
      tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)(acc * L::kAccStride);
      // TMEM is read kGrp 16-column chunks per round trip (one wait for several loads)
      constexpr int kGrp = kFused ? 1
                                  : (kW13Only ? (BN <= 32 ? 1 : 2) : (BN >= 64 ? (L::kAcc == 1 ? 2 : 4) : BN / 16));
      for (int cg = 16 * kGrp * half; cg < tw; cg += 16 * kGrp * kHalves) {
        uint32_t rg[kGrp][16];
        if (ok) {
#pragma unroll
          for (int h = 0; h < kGrp; ++h)
            if (cg + 16 * h < tw) tmem_ld16(d_tmem + lane_base + cg + 16 * h, rg[h]);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < kGrp; ++h) reg_fence16(rg[h]);
        }
#pragma unroll
        for (int h = 0; h < kGrp; ++h) {
          const int c0 = cg + 16 * h;
          if (c0 >= tw) break;
          const uint32_t(&r)[16] = rg[h];
          if (w13_item)
            epi_w13_chunk(r, xchg + half * 2 * 16 * 64, qd, lane, threadIdx.x - 128 - 128 * half, bar_id, ok, true,
                          c0, m, row0, nrows, q);
          else if (ok)
            epi_w2_chunk<!kFused>(r, qd, lane, c0, m, row0, nrows, q);
        }
      }
      if (kFused) __threadfence();                    // this lane's stores of the tile, before the count
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&acc_empty[acc]);
      if (kFused && lane == 0 && ok) {
        // publish the warp's part of the tile: per expert for a W13 tile (its h rows), in the grid
        // total for a W2 tile (the combine waits for all of them)
        __threadfence();
        atomicAdd(w13_item ? q.ready + e : q.ready + E, 1u);
      }
    }
    if (kFused && p2.out) {
      // ===================== the combine, after every W2 tile of the grid =====================
      // Unit u = (row t, 8 hidden features); the epilogue threads of all CTAs take units in turn.
      // A warp with units waits (one lane, bounded) until every W2 tile is counted, then folds
      // its rows exactly as the combine kernel does.
      constexpr int kEpiThreads = Threads<BN>::kEpiWarps * 32;
      const long long units = (long long)p2.T * (p2.H / 8);
      const long long gt = (long long)blockIdx.x * kEpiThreads + (threadIdx.x - 128);
      const long long gstride = (long long)gridDim.x * kEpiThreads;
      if (gt - lane < units) {
        // the unit's routing data come from the plan, written before this launch: pull them into L1
        // while the last down-projection tiles finish, so only the per-slot rows remain to fetch
        // (mode 3 holds them in shared memory)
        if (!kSelfPlan && gt < units) {
          const int tt = (int)(gt / (p2.H / 8));
          asm volatile("prefetch.global.L1 [%0];" ::"l"(p2.row_of_slot + (size_t)tt * p2.k));
          asm volatile("prefetch.global.L1 [%0];" ::"l"(p2.topk_w + (size_t)tt * p2.k));
        }
        uint32_t go = ok ? 1u : 0u;
        if (lane == 0 && go)
          go = wait_count_at_least(p2.ready + E, (uint32_t)(s_cum2[E] * Threads<BN>::kEpiWarps), kWaitLimitNs,
                                   abort_flag, p2.status) ? 1u : 0u;
        go = __shfl_sync(0xffffffffu, go, 0);
        __syncwarp();
        if (go)
          for (long long u = gt; u < units; u += gstride)
            combine_unit<true, kSelfPlan>(p2.y, kSelfPlan ? s_sw : p2.topk_w, kSelfPlan ? s_ros : p2.row_of_slot,
                                          (int)(u / (p2.H / 8)), (int)(u % (p2.H / 8)), p2.H, p2.k, p2.out, nullptr,
                                          nullptr, nullptr);
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // after an expired wait, TMA copies the producers issued may still be landing in shared
    // memory (their completion is only signalled on stage barriers whose other arrivals may never
    // come): give them time to land before the CTA's shared memory goes away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000) {
    }
  }
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, L::kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
// Token-tile width from the mean rows per expert. Wide tiles (MMA N up to MOE_WIDE_BN) are sized
// per expert inside the kernel: an N = 128 block-scaled MMA with its scale copies occupies the
// tensor core about as long as an N = 256 one, so fewer, wider tiles raise the math rate.
static int pick_bn(const moe_shape* s) {
  const double avg = (double)s->T * s->k / s->E;
  if (avg <= 16) return 16;
  if (avg <= 32) return 32;
  if (avg <= 64) return 64;
  return MOE_WIDE_BN;
}

template <int BN, int MODE>
static int launch_gemm_bn(const CUtensorMap& tm, const CUtensorMap& tmb, const CUtensorMap& tm2, const GemmParams& gp,
                          const GemmParams& gp2, long long max_items, cudaStream_t st) {
  using L = Smem<BN>;
  auto kern = grouped_gemm_kernel<BN, MODE>;
  const int smem = L::total(gp.E, MODE >= 2, MODE == 3 ? gp.T * gp.k : 0);
  const int smem_max = MODE == 3 ? L::total(kSelfPlanMaxE, true, kSelfPlanMaxT * kMaxK) : L::total(kMaxE, MODE == 2);
  if (ensure_smem_limit((const void*)kern, smem_max)) return MOE_ERR_CUDA;
  // persistent grid: as many CTAs as fit on the GPU at once (smem depends on E); the one-launch
  // W13 + W2 modes rely on every CTA being resident
  const int occ = ctas_per_sm_by_smem((size_t)smem, L::kCtasPerSm);
  const long long grid = std::min<long long>(max_items, (long long)occ * num_sms());
  if (grid <= 0) return MOE_OK;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(Threads<BN>::kCount), (size_t)smem, st, tm, tmb, tm2, gp, gp2);
}

static int weight_tmap(CUtensorMap* tm, const moe_shape* s, const uint8_t* codes, const GemmParams& gp, int box_tiles) {
  const long long tiles = (long long)s->E * gp.MT * gp.KC;
  return gp.a_fp8 ? make_weight_tmap_fp8(tm, codes, tiles, box_tiles) : make_weight_tmap(tm, codes, tiles, box_tiles);
}

template <bool W13>
static int launch_gemm(const moe_shape* s, const uint8_t* codes, const GemmParams& gp, cudaStream_t st) {
  const long long slots = (long long)s->T * s->k;
  // TMA row coordinates of the packed weights are 32-bit: 128 rows per tile
  if ((long long)s->E * gp.MT * gp.KC * 128 >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int bn = pick_bn(s);
  // a wide down projection with a short K keeps each weight panel resident while the expert's token
  // tiles stream past it (gemm_ws.cu); with a long K, and for the gate/up GEMM, one-CTA wide tiles
  if (!W13 && bn > 64 && ws_down_supported(s)) return launch_gemm_ws(s, codes, gp, st);
  CUtensorMap tm;
  const int box_tiles = (bn <= 32) ? Smem<16>::KT : (bn <= 64 ? Smem<64>::KT : Smem<MOE_WIDE_BN>::KT);
  int rc0 = weight_tmap(&tm, s, codes, gp, box_tiles);
  if (rc0) return rc0;
  // activation operand of the wide token tile as a TMA tensor: [T*k plan rows, K] bytes, boxes of
  // bn plan rows (W13: the plan-order copy of xq; W2: hq)
  CUtensorMap tmb = tm;
  const long long max_items = (long long)gp.MT * ((slots + bn - 1) / bn + std::min<long long>(s->E, slots));
  if (bn >= 128) {
    const int rc = make_act_tmap(&tmb, gp.bq, gp.b_row_bytes, slots, bn);
    if (rc) return rc;
  }
  constexpr int M = W13 ? 1 : 0;
  switch (bn) {
    case 16: return launch_gemm_bn<16, M>(tm, tmb, tm, gp, gp, max_items, st);
    case 32: return launch_gemm_bn<32, M>(tm, tmb, tm, gp, gp, max_items, st);
    case 64: return launch_gemm_bn<64, M>(tm, tmb, tm, gp, gp, max_items, st);
    default: return launch_gemm_bn<MOE_WIDE_BN, M>(tm, tmb, tm, gp, gp, max_items, st);
  }
}

// Copies the quantised activation rows (codes and scale bytes) into plan order: plan row p gets
// token slot_of_row[p] / k. Only the first offsets[E] rows are live; the rest are left untouched.
__global__ void gather_plan_rows_kernel(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xs, int H,
                                        const int32_t* __restrict__ slot_of_row, const int32_t* __restrict__ offsets,
                                        int E, int k, int max_rows, uint8_t* __restrict__ xqp,
                                        uint8_t* __restrict__ xsp) {
  pdl_trigger();
  pdl_wait();
  const int S = min(offsets[E], max_rows);
  const int q16 = H / 16, s4 = H / 128;          // 16-byte code chunks and 4-byte scale words per row
  const int per_row = q16 + s4;
  const long long n = (long long)S * per_row;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int prow = (int)(i / per_row), j = (int)(i % per_row);
    const int t = slot_of_row[prow] / k;
    if (j < q16) {
      reinterpret_cast<uint4*>(xqp + (size_t)prow * H)[j] = __ldg(reinterpret_cast<const uint4*>(xq + (size_t)t * H) + j);
    } else {
      const int w = j - q16;
      reinterpret_cast<uint32_t*>(xsp + (size_t)prow * (H / 32))[w] =
          __ldg(reinterpret_cast<const uint32_t*>(xs + (size_t)t * (H / 32)) + w);
    }
  }
}

bool w13_wants_plan_rows(const moe_shape* s) { return pick_bn(s) >= 128; }

// Parameters of the gate/up GEMM reading xq / xs (token rows, or plan rows with plan_rows).
static GemmParams w13_params(const moe_shape* s, const uint8_t* xq, const uint8_t* xs, bool plan_rows,
                             const uint8_t* w13, const uint8_t* w13s, const int32_t* offsets,
                             const int32_t* slot_of_row, uint8_t* hq, uint8_t* hs, float* dbg, uint32_t* status,
                             bool fp8_weights) {
  GemmParams gp{};
  gp.a_fp8 = fp8_weights ? 1 : 0;
  gp.bq = xq;
  gp.bs = xs;
  gp.b_plan_rows = plan_rows ? 1 : 0;
  gp.b_row_bytes = s->H;
  gp.b_scale_pitch = s->H / 32;
  gp.a_codes = w13;
  gp.a_scales = w13s;
  gp.offsets = offsets;
  gp.slot_of_row = slot_of_row;
  gp.E = s->E;
  gp.k = s->k;
  gp.K = s->H;
  gp.KC = s->H / kTileK;
  gp.MT = s->I / 64;
  gp.I = s->I;
  gp.H = s->H;
  gp.hq = hq;
  gp.hs = hs;
  gp.hs_pitch = hs_pitch(s->I);
  gp.dbg = dbg;
  gp.status = status;
  return gp;
}

// Parameters of the down projection reading hq / hs (plan rows) into plan-order y.
static GemmParams w2_params(const moe_shape* s, const uint8_t* hq, const uint8_t* hs, const uint8_t* w2,
                            const uint8_t* w2s, const int32_t* offsets, const int32_t* slot_of_row, float* y,
                            uint32_t* status, bool fp8_weights) {
  GemmParams gp{};
  gp.a_fp8 = fp8_weights ? 1 : 0;
  gp.bq = hq;
  gp.bs = hs;
  gp.b_row_bytes = s->I;
  gp.b_scale_pitch = hs_pitch(s->I);
  gp.a_codes = w2;
  gp.a_scales = w2s;
  gp.offsets = offsets;
  gp.slot_of_row = slot_of_row;
  gp.E = s->E;
  gp.k = s->k;
  gp.K = s->I;
  gp.KC = ceil_div(s->I, kTileK);
  gp.MT = s->H / 128;
  gp.I = s->I;
  gp.H = s->H;
  gp.y = y;
  gp.status = status;
  return gp;
}

int launch_w13(const moe_shape* s, const uint8_t* xq, const uint8_t* xs, const uint8_t* w13, const uint8_t* w13s,
               const int32_t* offsets, const int32_t* slot_of_row, uint8_t* hq, uint8_t* hs, float* dbg,
               uint32_t* status, uint8_t* xq_plan, uint8_t* xs_plan, bool plan_rows_ready, cudaStream_t st,
               bool fp8_weights) {
  if (s->T == 0) return MOE_OK;
  bool plan_rows = false;
  if (plan_rows_ready) {
    // the activation rows already sit in plan order (wide tiles read them with TMA boxes, narrow
    // tiles gather plan row p for column p)
    xq = xq_plan;
    xs = xs_plan;
    plan_rows = true;
  } else if (pick_bn(s) >= 128) {
    // wide tiles read the token operand in plan order with TMA boxes: gather it once
    const long long n = (long long)s->T * s->k * (s->H / 16 + s->H / 128);
    const int blocks = (int)std::min<long long>((n + 255) / 256, (long long)num_sms() * 8);
    const int rc = launch_pdl(gather_plan_rows_kernel, dim3(blocks), dim3(256), 0, st, xq, xs, s->H, slot_of_row,
                              offsets, s->E, s->k, s->T * s->k, xq_plan, xs_plan);
    if (rc) return rc;
    xq = xq_plan;
    xs = xs_plan;
    plan_rows = true;
  }
  const GemmParams gp = w13_params(s, xq, xs, plan_rows, w13, w13s, offsets, slot_of_row, hq, hs, dbg, status,
                                   fp8_weights);
  return launch_gemm<true>(s, w13, gp, st);
}

int launch_w2(const moe_shape* s, const uint8_t* hq, const uint8_t* hs, const uint8_t* w2, const uint8_t* w2s,
              const int32_t* offsets, const int32_t* slot_of_row, float* y, uint32_t* status,
              cudaStream_t st, bool fp8_weights) {
  if (s->T == 0) return MOE_OK;
  const GemmParams gp = w2_params(s, hq, hs, w2, w2s, offsets, slot_of_row, y, status, fp8_weights);
  return launch_gemm<false>(s, w2, gp, st);
}

bool fused_gemms_supported(const moe_shape* s) { return pick_bn(s) <= 32; }

int launch_w13_w2_fused(const moe_shape* s, const uint8_t* xq, const uint8_t* xs, const uint8_t* w13,
                        const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, const int32_t* offsets,
                        const int32_t* slot_of_row, uint8_t* hq, uint8_t* hs, float* dbg, float* y, uint32_t* status,
                        uint32_t* ready, cudaStream_t st, const float* topk_w, const int32_t* row_of_slot,
                        uint16_t* out, const SelfPlanArgs* sp) {
  if (s->T == 0) return MOE_OK;
  const int bn = pick_bn(s);
  if (bn > 32 || !ready) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (sp && (!out || !self_plan_supported(s))) return MOE_ERR_UNSUPPORTED_SHAPE;
  GemmParams g13 = w13_params(s, xq, xs, false, w13, w13s, offsets, slot_of_row, hq, hs, dbg, status, false);
  GemmParams g2 = w2_params(s, hq, hs, w2, w2s, offsets, slot_of_row, y, status, false);
  g13.ready = ready;
  g2.ready = ready;
  if (out) {
    if (!topk_w || !row_of_slot) return MOE_ERR_INVALID_ARG;
    g2.topk_w = topk_w;
    g2.row_of_slot = row_of_slot;
    g2.out = out;
    g2.T = s->T;
  }
  if (sp) {
    g13.T = s->T;
    g13.sel = sp->sel;
    g13.dead = sp->dead;
    g13.plan_topk_idx = sp->topk_idx;
    g13.plan_topk_w = sp->topk_w;
    g13.plan_counts = sp->counts;
    g13.plan_offsets = sp->offsets;
    g13.plan_slot_of_row = sp->slot_of_row;
    g13.plan_row_of_slot = sp->row_of_slot;
  }
  if ((long long)s->E * std::max(g13.MT * g13.KC, g2.MT * g2.KC) * 128 >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap t13, t2;
  int rc = weight_tmap(&t13, s, w13, g13, Smem<16>::KT);
  if (!rc) rc = weight_tmap(&t2, s, w2, g2, Smem<16>::KT);
  if (rc) return rc;
  const long long slots = (long long)s->T * s->k;
  const long long max_items = (long long)(g13.MT + g2.MT) * ((slots + bn - 1) / bn + std::min<long long>(s->E, slots));
  // a self-routed batch (at most kSelfPlanMaxT rows, k <= E) has T k / E <= kSelfPlanMaxT rows per
  // expert on average: always 16-row tiles
  if (sp) return bn == 16 ? launch_gemm_bn<16, 3>(t13, t13, t2, g13, g2, max_items, st) : MOE_ERR_UNSUPPORTED_SHAPE;
  return bn == 16 ? launch_gemm_bn<16, 2>(t13, t13, t2, g13, g2, max_items, st)
                  : launch_gemm_bn<32, 2>(t13, t13, t2, g13, g2, max_items, st);
}

}  // namespace moe
