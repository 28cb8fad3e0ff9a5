// Grouped block-scaled GEMMs of the routed experts on CTA pairs (tcgen05 .cta_group::2), for wide
// (prefill) token tiles. Built and parity-checked for both GEMMs (same results as every other tile
// kind); the layer dispatches neither to it: the gate/up GEMM runs faster on one-CTA tiles and the
// short-K down projection on weight-stationary tiles (gemm_ws.cu).
//
// "New Deepseek 4.1 flash recipe", post 6 "How it works" items 1-2: FP8 activations x FP4 weights
// through a block-scaled MMA (kind::mxf8f6f4); prefill rasterises weights larger than L2 in panels.
// Post 4 "Fenced pipeline stages": a stage is refilled only after every read of it completed.
//
// A work item is (expert, pair of weight panels, token tile): one MMA of M = 256 weight rows (the
// even CTA's panel 2mp and the odd CTA's panel 2mp + 1, 128 packed rows each) by N = tw token
// columns (the expert's rows spread evenly over its tiles, at most 224), K looped in 128-element
// chunks, never split. Each CTA stages its own weight panel, HALF of the tile's token rows (the
// MMA's B columns are split between the two SMs) and the scale bytes of all tw columns; each
// shared-memory byte a CTA holds is therefore read by the tensor cores of both SMs, which halves the
// token-operand traffic per SM against one-CTA tiles. A row's result is the same as on any other
// tile kind: same K order, same fp32 accumulation per column, the same epilogue code (gemm.cuh).
//
// Roles (both CTAs of a pair run the same code; 384 threads with one pair per SM pair, 256 with
// two):
//   warp 0      weight TMA (FP4 tile unpacked to 8-bit containers) and its 512-byte scale block
//   warp 1      token TMA (one box of tw/2 plan rows) and the scale bytes of all tw columns
//               (the weight and token boxes of both CTAs complete on the even CTA's stage barrier)
//   warp 2      even CTA: tcgen05.cp of the scale blocks and the pair's MMAs, commits multicast to
//               both CTAs' stage and accumulator barriers; odd CTA: tells the even CTA when its
//               scale bytes for a stage have landed. Both: the pair's TMEM allocation.
//   warps 4-11  epilogue of the CTA's 128 accumulator rows (two sets of four warps, alternating
//               column groups): SwiGLU + MXFP8 requant (W13) or plan-order fp32 rows (W2); each set
//               tells the even CTA when an accumulator slot is free again.
// Every wait is bounded; after an expired wait a CTA records a code in the status word, turns the
// rest of its loops into no-ops that still meet at the named barriers, and both CTAs meet at a final
// cluster barrier before the pair's TMEM is released.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "gemm.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

// Tile configurations of the pair kernel: token-tile width BN (MMA N across the pair), pipeline
// stages, and pairs resident per SM pair (1: two accumulator slots, 8 epilogue warps; 2: one
// accumulator slot per CTA, 4 epilogue warps, the other pair's MMAs covering each epilogue).
template <int BN_, int STAGES, int CTAS>
struct PairCfg {
  static constexpr int BN = BN_;
  static constexpr int kHalfRows = BN / 2;                 // token rows each CTA stages
  static constexpr int kStages = STAGES;
  static constexpr int kCtasPerSm = CTAS;
  static constexpr int kAcc = CTAS == 1 ? 2 : 1;
  static constexpr int kEpiWarps = CTAS == 1 ? 8 : 4;
  static constexpr int kSets = kEpiWarps / 4;              // epilogue sets of four warps
  static constexpr int kThreads = 128 + 32 * kEpiWarps;
  static constexpr int kTileA = 16384;                     // one 128 x 128 weight tile in 8-bit containers
  static constexpr int kTileB = kHalfRows * 128;           // BN/2 token rows x 128 FP8
  static constexpr int kSfbAtoms = (BN + 127) / 128;       // B scale atoms (128 token columns each)
  static constexpr int kSfChunk = 512 + 512 * kSfbAtoms;
  static constexpr int kStageBytes = (kTileA + kTileB + kSfChunk + 1023) / 1024 * 1024;
  static constexpr int kTiles = kStages * kStageBytes;
  static constexpr int kXchg = kSets * 2 * 16 * 64 * 4;    // per set: (gate + up) [16][64] fp32
  static constexpr int kMisc = 1024;
  static constexpr int kFixed = 1024 + kTiles + kXchg + kMisc;
  static int total(int E) { return kFixed + (int)align_up((size_t)(E + 1) * 8, 16); }
  // TMEM (same columns in both CTAs): kAcc accumulator slots of BN columns, then one scale slot per
  // stage (4 columns of A scales, 4 per B atom)
  static constexpr int kAccStride = BN;
  static constexpr int kSfCol = kAcc * BN;
  static constexpr int kSfSlot = 4 + 4 * kSfbAtoms;
  static constexpr int kTmemCols = 512 / CTAS;
  static_assert(kSfCol + kStages * kSfSlot <= kTmemCols, "TMEM columns");
  static_assert(BN % 32 == 0 && BN <= 256, "pair tile width");
  static_assert(CTAS == 1 || CTAS == 2, "pairs per SM pair");
  static_assert(kFixed + (kMaxE + 1) * 8 + 16 <= (CTAS == 1 ? 227 * 1024 : 113 * 1024),
                "shared memory per CTA at the largest E");
};

template <bool W13, class Pair>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Pair::kThreads, Pair::kCtasPerSm)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                             const GemmParams p) {
  constexpr int S = Pair::kStages;
  constexpr int NACC = Pair::kAcc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = base;
  float* xchg = reinterpret_cast<float*>(base + Pair::kTiles);
  uint8_t* misc = base + Pair::kTiles + Pair::kXchg;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;          // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2], arrived on by both CTAs' epilogues (used in the even CTA)
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  int* s_off = reinterpret_cast<int*>(misc + Pair::kMisc);   // expert offsets [E+1]
  int* s_cum = s_off + (p.E + 1);                            // first work item of each expert [E+1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();                   // 0: issues the pair's MMAs
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int E = p.E;
  const int MP = (p.MT + 1) >> 1;                            // panel pairs per expert

  // ---- prologue: barriers and the pair's TMEM (overlaps the previous kernel), then the plan ----
  pdl_trigger();
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      // weight producer + 32 token-producer lanes (+ the odd CTA's relay, in the even CTA)
      mbar_init(&full[s], 1 + 32 + (rank == 0 ? 1 : 0));
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 2 * Pair::kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, Pair::kTmemCols);
    tmem_relinquish_pair();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += Pair::kThreads) s_off[i] = p.offsets[i];
  __syncthreads();
  if (warp == 0) {
    // work items per expert: ceil(count / BN) token tiles x MP panel pairs (warp prefix sum)
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int local = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) local += (s_off[e + 1] - s_off[e] + Pair::BN - 1) / Pair::BN;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      s_cum[e] = run * MP;
      run += (s_off[e + 1] - s_off[e] + Pair::BN - 1) / Pair::BN;
    }
    if (lane == 31) s_cum[E] = incl * MP;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // both CTAs' barriers exist before either arrives on the other's
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = s_cum[E];

  // work item w -> expert e, panel pair mp, token tile nt of width tw (the expert's rows spread
  // evenly over ceil(count / BN) tiles, rounded up to 32 so each CTA's half is a multiple of 16)
  auto decode = [&](int w, int& e, int& mp, int& row0, int& nrows, int& tw) {
    e = find_expert(s_cum, E, w);
    const int cnt = s_off[e + 1] - s_off[e];
    const int ntiles = (cnt + Pair::BN - 1) / Pair::BN;
    tw = min(Pair::BN, ((cnt + ntiles - 1) / ntiles + 31) / 32 * 32);
    const int local = w - s_cum[e];
    mp = local / ntiles;
    const int nt = local - mp * ntiles;
    row0 = s_off[e] + nt * tw;
    nrows = min(tw, cnt - nt * tw);
  };

  if (warp == 0) {
    // ===================== TMA producer: this CTA's weight panel =====================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t tile_bytes = p.a_fp8 ? 2 * kTileCodeBytes : kTileCodeBytes;
      // the weight and token boxes of BOTH CTAs complete on the even CTA's stage barrier: its
      // producer announces all of them; the odd CTA's own barrier only counts its scale copies
      const uint32_t leader_full = mapa_shared(&full[0], 0);
      const uint32_t expect = rank == 0 ? 2 * (tile_bytes + Pair::kTileB) + kTileScaleBytes : kTileScaleBytes;
      for (int w = pair; w < total && ok; w += npairs) {
        int e, mp, row0, nrows, tw;
        decode(w, e, mp, row0, nrows, tw);
        // the odd CTA of an expert's last pair when MT is odd loads a real panel (the last one)
        // so the MMA reads defined data; its rows are never stored
        const int m = min(2 * mp + (int)rank, p.MT - 1);
        const int tile0 = (e * p.MT + m) * p.KC;
        for (int kc = 0; kc < p.KC; ++kc) {
          if (!mbar_wait(&empty[stage], phase ^ 1, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_EMPTY)) {
            ok = false;
            break;
          }
          uint8_t* sA = tiles + stage * Pair::kStageBytes;
          uint8_t* sSFA = sA + Pair::kTileA + Pair::kTileB;
          mbar_arrive_expect_tx(&full[stage], expect);
          tma_load_2d_pair(sA, &tmap_a, 0, (tile0 + kc) * 128, leader_full + (uint32_t)(stage * 8));
          bulk_load(sSFA, p.a_scales + (size_t)(tile0 + kc) * kTileScaleBytes, kTileScaleBytes, &full[stage]);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ===================== TMA producer: this CTA's half of the token rows =====================
    // lane 0 loads one box of BN/2 plan rows starting at the CTA's half of the tile (rows past the
    // tile belong to the next tile or expert, or are TMA zero fill, and are never stored); the lanes
    // write the scale atoms of the WHOLE tile, which each SM's MMA reads from its own Tensor
    // Memory, with 16-byte shared stores. The chunks stream in order (items w, K-chunks kc); a
    // chunk's scale words are loaded one chunk ahead, before the previous chunk's are stored.
    constexpr int NA = Pair::kSfbAtoms;
    const uint32_t leader_full = mapa_shared(&full[0], 0);
    int w = pair, kn = 0;
    int e = 0, mp = 0, row0 = 0, nrows = 0, tw = 0;
    if (w < total) decode(w, e, mp, row0, nrows, tw);
    auto next_chunk = [&](int& r0, int& nr, int& tw0, int& kc) {   // the chunk at the cursor, then advance
      if (w >= total) return false;
      r0 = row0;
      nr = nrows;
      tw0 = tw;
      kc = kn;
      if (++kn == p.KC) {
        kn = 0;
        w += npairs;
        if (w < total) decode(w, e, mp, row0, nrows, tw);
      }
      return true;
    };
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int r0 = 0, nr = 0, tw0 = 0, kc = 0;
    bool have = next_chunk(r0, nr, tw0, kc);
    ScaleLines<NA> sl;
    if (have) load_scale_lines(sl, p.bs, p.b_scale_pitch, r0, nr, kc, lane);
    while (have) {
      int r1 = 0, nr1 = 0, tw1 = 0, kc1 = 0;
      const bool have1 = next_chunk(r1, nr1, tw1, kc1);
      ScaleLines<NA> sl1;
      if (have1) load_scale_lines(sl1, p.bs, p.b_scale_pitch, r1, nr1, kc1, lane);
      if (ok) ok = warp_wait(&empty[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_EMPTY);
      if (ok) {
        uint8_t* sB = tiles + stage * Pair::kStageBytes + Pair::kTileA;
        uint8_t* sSFB = sB + Pair::kTileB + 512;
        const int brow = r0 + (int)rank * (tw0 >> 1);
        if (lane == 0) tma_load_2d_pair(sB, &tmap_b, kc * 128, brow, leader_full + (uint32_t)(stage * 8));
        store_scale_lines(sl, sSFB, lane);
        fence_async_smem();
        mbar_arrive(&full[stage]);
      }
      if (++stage == S) { stage = 0; phase ^= 1; }
      have = have1;
      r0 = r1;
      nr = nr1;
      tw0 = tw1;
      kc = kc1;
      sl = sl1;
    }
  } else if (warp == 2) {
    if (lane == 0 && rank == 0) {
      // ===================== the pair's MMA issuer (even CTA) =====================
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int w = pair; w < total && ok; w += npairs, ++it) {
        int e, mp, row0, nrows, tw;
        decode(w, e, mp, row0, nrows, tw);
        const uint32_t idesc_base = idesc_mxf8f6f4(p.a_fp8 ? 0 : 5 /*weights E4M3 or E2M1*/, 0 /*E4M3*/, 256, tw, 0, 0);
        const int acc = (NACC == 2) ? (it & 1) : 0;
        const int use = (NACC == 2) ? (it >> 1) : it;
        if (use > 0 && !mbar_wait_cluster(&acc_empty[acc], (use - 1) & 1, kWaitLimitNs, abort_flag, p.status,
                                          DEV_TIMEOUT_DRAIN)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * Pair::kAccStride);
        for (int kc = 0; kc < p.KC; ++kc) {
          if (!mbar_wait_cluster(&full[stage], phase, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_FULL)) {
            ok = false;
            break;
          }
          fence_async_smem();
          tc_fence_after();
          uint8_t* sA = tiles + stage * Pair::kStageBytes;
          uint8_t* sB = sA + Pair::kTileA;
          uint8_t* sSFA = sB + Pair::kTileB;
          uint8_t* sSFB = sSFA + 512;
          const uint32_t tsfa = tmem + Pair::kSfCol + stage * Pair::kSfSlot;
          const uint32_t tsfb = tsfa + 4;
          tc_cp_32x128b_warpx4_pair(tsfa, smem_desc(smem_u32(sSFA), 16, 128, 0));
          for (int q = 0; q * 128 < tw; ++q)
            tc_cp_32x128b_warpx4_pair(tsfb + 4 * q, smem_desc(smem_u32(sSFB + q * 512), 16, 128, 0));
          const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
          const int nk = min(4, (p.K - kc * 128) / 32);
          for (int kb = 0; kb < nk; ++kb) {
            const uint64_t ad = smem_desc(a0 + kb * 32, 16, 1024, 2);
            const uint64_t bd = smem_desc(b0 + kb * 32, 16, 1024, 2);
            const uint32_t id = idesc_base | ((uint32_t)kb << 4) | ((uint32_t)kb << 29);
            mma_mxf8f6f4_pair(d_tmem, ad, bd, id, tsfa, tsfb, (kc > 0 || kb > 0) ? 1u : 0u);
          }
          tc_commit_pair_mc(&empty[stage], 0x3);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair_mc(&acc_full[acc], 0x3);
      }
      // every MMA and scale copy issued for the pair has completed before either CTA releases its
      // shared memory or the pair's TMEM (this wait does not take the abort shortcut)
      tc_commit_pair_mc(drain, 0x1);
      mbar_wait(drain, 0, kWaitLimitNs, nullptr, p.status, DEV_TIMEOUT_DRAIN);
    } else if (lane == 0) {
      // ===================== relay (odd CTA): "my scale bytes for this stage have landed" =====================
      // (its weight and token boxes complete on the even CTA's barrier directly; only the small
      // scale copies, which complete on this CTA's barrier, are relayed)
      const uint32_t leader_full = mapa_shared(&full[0], 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = pair; w < total && ok; w += npairs) {
        for (int kc = 0; kc < p.KC; ++kc) {
          if (!mbar_wait(&full[stage], phase, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_FULL)) {
            ok = false;
            break;
          }
          fence_async_smem();          // the scale bytes were written by cp.async (generic proxy)
          mbar_arrive_cluster(leader_full + (uint32_t)(stage * 8));
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ===================== epilogue (warp w -> TMEM lanes 32 (w % 4)) =====================
    // With two sets, warps 4-7 take the even 16 kGrp-column groups of a tile and warps 8-11 the odd
    // ones, each set with its own exchange buffer and named barrier.
    const int q = (warp - 4) & 3;
    const int half = (warp - 4) >> 2;
    const uint32_t bar_id = 1 + 2 * half;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const uint32_t leader_acc_empty = mapa_shared(&acc_empty[0], 0);
    int it = 0;
    bool ok = true;
    for (int w = pair; w < total; w += npairs, ++it) {
      int e, mp, row0, nrows, tw;
      decode(w, e, mp, row0, nrows, tw);
      const int m = 2 * mp + (int)rank;
      const bool store = m < p.MT;
      const int acc = (NACC == 2) ? (it & 1) : 0;
      const int use = (NACC == 2) ? (it >> 1) : it;
      if (ok) ok = warp_wait(&acc_full[acc], use & 1, abort_flag, p.status, DEV_TIMEOUT_ACCUM);
      tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)(acc * Pair::kAccStride);
      constexpr int kGrp = W13 ? 2 : 4;
      for (int cg = 16 * kGrp * half; cg < tw; cg += 16 * kGrp * Pair::kSets) {
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
          if constexpr (W13)
            epi_w13_chunk(rg[h], xchg + half * 2 * 16 * 64, q, lane, threadIdx.x - 128 - 128 * half, bar_id, ok,
                          store, c0, m, row0, nrows, p);
          else if (ok && store)
            epi_w2_chunk<true>(rg[h], q, lane, c0, m, row0, nrows, p);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && ok) {
        if (rank == 0)
          mbar_arrive(&acc_empty[acc]);
        else
          mbar_arrive_cluster(leader_acc_empty + (uint32_t)(acc * 8));
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // after an expired wait, TMA copies issued by this CTA may still be landing in its shared
    // memory: give them time before the CTA's shared memory goes away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000) {
    }
  }
  // the pair's MMAs read both CTAs' shared memory and write both CTAs' TMEM: neither CTA leaves
  // (or releases the pair's columns) before the other is done
  cluster_sync_all();
  tc_fence_after();
  if (warp == 2) tmem_dealloc_pair(tmem, Pair::kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
template <bool W13, class Pair>
static int launch_pair_t(const moe_shape* s, const uint8_t* codes, const GemmParams& gp, cudaStream_t st) {
  const long long slots = (long long)s->T * s->k;
  if ((long long)s->E * gp.MT * gp.KC * 128 >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap tm, tmb;
  const long long tiles = (long long)s->E * gp.MT * gp.KC;
  int rc = gp.a_fp8 ? make_weight_tmap_fp8(&tm, codes, tiles, 1) : make_weight_tmap(&tm, codes, tiles, 1);
  if (rc) return rc;
  rc = make_act_tmap(&tmb, gp.bq, gp.b_row_bytes, slots, Pair::kHalfRows);
  if (rc) return rc;
  auto kern = grouped_gemm_pair_kernel<W13, Pair>;
  if (ensure_smem_limit((const void*)kern, Pair::total(kMaxE))) return MOE_ERR_CUDA;
  const int MP = (gp.MT + 1) / 2;
  const long long max_items = (long long)MP * ((slots + Pair::BN - 1) / Pair::BN + std::min<long long>(s->E, slots));
  const int occ = ctas_per_sm_by_smem((size_t)Pair::total(gp.E), Pair::kCtasPerSm);
  const long long pairs = std::min<long long>(max_items, (long long)occ * (num_sms() / 2));
  if (pairs <= 0) return MOE_OK;
  return launch_pdl(kern, dim3((unsigned)(2 * pairs)), dim3(Pair::kThreads), (size_t)Pair::total(gp.E), st, tm, tmb,
                    gp);
}

// The configuration in use: tiles of up to 192 columns, 3 stages, two pairs per SM pair (measured
// fastest of {224 columns, 5 stages, one pair}, {192, 6, one pair}, {192, 3, two pairs}: the
// second pair keeps each SM's tensor core fed while the first waits on its stages).
using PairTile = PairCfg<192, 3, 2>;

int launch_gemm_pair(const moe_shape* s, const uint8_t* codes, const GemmParams& gp, bool w13, cudaStream_t st) {
  return w13 ? launch_pair_t<true, PairTile>(s, codes, gp, st) : launch_pair_t<false, PairTile>(s, codes, gp, st);
}

}  // namespace moe
