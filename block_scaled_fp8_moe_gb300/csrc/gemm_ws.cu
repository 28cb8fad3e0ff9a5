// Down projection with a short K on weight-stationary tiles (tcgen05, one CTA per SM).
//
// "New Deepseek 4.1 flash recipe", post 6 "How it works" items 1-2 (FP8 activations x FP4 weights
// through kind::mxf8f6f4; panels of weights); TP4 serving profile README, settings table "Experts"
// row (per-slot buffer: this kernel writes its rows, the combine sums them in a fixed order).
//
// When the down projection's K (the expert intermediate size I) is short, a whole 128-row weight
// panel, all its K-chunks unpacked to 8-bit containers, fits in shared memory (I = 576: 5 chunks,
// 80 KB). A work unit is then (expert e, panel m, a block of up to kTilesPerUnit token tiles of e):
// the panel and its scale blocks are loaded once per unit and stay resident while the unit's token
// tiles stream past them, so each tile moves only its token rows instead of the panel again. CTAs
// running at the same time take different panels of the same token tiles (panel fastest), which
// therefore come from L2. A row's result is the same as on the other tile kinds: same K order,
// same per-column fp32 accumulation, same epilogue (gemm.cuh).
//
// Roles (384 threads):
//   warp 0      TMA of the unit's weight panel (KC tiles) and its scale blocks into the resident
//               region, each K-chunk as soon as the previous unit's last MMAs on it are done (one
//               barrier pair per resident chunk)
//   warp 1      per (tile, K-chunk): one TMA box of plan rows (lane 0) and the scale atoms of the
//               tile's columns (every lane: plain loads, 16-byte shared stores) into a ring of stages
//   warp 2      TMEM owner and MMA issuer: the unit's A scales into resident TMEM columns as its
//               chunks land, then per K-chunk the stage's B scales and four K = 32 MMAs; commits
//               release stages, accumulators and, after the unit's last tile, each resident chunk
//   warps 4-11  epilogue: plan-order fp32 rows of the per-slot buffer (two sets of four warps,
//               alternating column groups; two accumulator slots)
// Every wait is bounded; after an expired wait the CTA records a code in the status word and its
// remaining loops do nothing but meet at the named barriers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "gemm.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

struct Ws {
  static constexpr int BN = 224;                        // widest token tile (MMA N)
  static constexpr int kKcMax = 6;                      // resident K-chunks (I <= 768)
  static constexpr int kTilesPerUnit = 8;
  static constexpr int kStages = 4;
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = 128 + 32 * kEpiWarps;
  static constexpr int kTileA = 16384;                  // 128 x 128 weight tile in 8-bit containers
  static constexpr int kTileB = BN * 128;               // BN plan rows x 128 FP8
  static constexpr int kSfb = 512 * ((BN + 127) / 128); // B scale atoms of one K-chunk
  static constexpr int kResA = kKcMax * kTileA;
  static constexpr int kResSfa = kKcMax * 512;
  static constexpr int kStageBytes = (kTileB + kSfb + 1023) / 1024 * 1024;
  static constexpr int kTiles = kResA + kResSfa + kStages * kStageBytes;
  static constexpr int kMisc = 1024;
  static constexpr int kFixed = 1024 + kTiles + kMisc;
  static int total(int E) { return kFixed + (int)align_up((size_t)(E + 1) * 8, 16); }
  // TMEM: two accumulator slots, the unit's A scales (4 columns per K-chunk), a ring of B scales
  static constexpr int kAccStride = BN;
  static constexpr int kSfaCol = 2 * BN;
  static constexpr int kSfbCol = kSfaCol + 4 * kKcMax;
  static constexpr int kSfbSlot = 4 * ((BN + 127) / 128);
  static constexpr int kTmemCols = 512;
  static_assert(kSfbCol + kStages * kSfbSlot <= kTmemCols, "TMEM columns");
  static_assert(kFixed + (kMaxE + 1) * 8 + 16 <= 227 * 1024, "shared memory per CTA at the largest E");
  static_assert(kResA % 1024 == 0 && kResSfa % 1024 == 0 && kStageBytes % 1024 == 0, "1 KB aligned regions");
};

__global__ void __launch_bounds__(Ws::kThreads, 1)
    grouped_gemm_ws_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                           const GemmParams p) {
  constexpr int S = Ws::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* resA = base;                                  // [kKcMax][128 rows x 128 B]
  uint8_t* resSfa = base + Ws::kResA;                    // [kKcMax][512 B]
  uint8_t* stages = resSfa + Ws::kResSfa;                // [S][token box | B scales]
  uint8_t* misc = base + Ws::kTiles;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;                        // [2]
  uint64_t* acc_empty = acc_full + 2;                    // [2]
  uint64_t* a_full = acc_empty + 2;                      // [kKcMax]: one per resident K-chunk
  uint64_t* a_empty = a_full + Ws::kKcMax;               // [kKcMax]
  uint64_t* drain = a_empty + Ws::kKcMax;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  int* s_off = reinterpret_cast<int*>(misc + Ws::kMisc);   // expert offsets [E+1]
  int* s_cum = s_off + (p.E + 1);                          // first unit of each expert [E+1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int KC = p.KC;

  pdl_trigger();
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + 32);                       // lane 0's expect-tx arrival + 32 scale-store arrivals
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], Ws::kEpiWarps);
    }
    for (int kc = 0; kc < Ws::kKcMax; ++kc) {
      mbar_init(&a_full[kc], 1);
      mbar_init(&a_empty[kc], 1);
    }
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, Ws::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += Ws::kThreads) s_off[i] = p.offsets[i];
  __syncthreads();
  if (warp == 0) {
    // units per expert: MT panels x ceil(tiles / kTilesPerUnit) blocks of token tiles
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int local = 0;
    auto blocks_of = [&](int e) {
      const int nt = (s_off[e + 1] - s_off[e] + Ws::BN - 1) / Ws::BN;
      return (nt + Ws::kTilesPerUnit - 1) / Ws::kTilesPerUnit;
    };
    for (int e = e0; e < min(E, e0 + per); ++e) local += blocks_of(e);
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      s_cum[e] = run * p.MT;
      run += blocks_of(e);
    }
    if (lane == 31) s_cum[E] = incl * p.MT;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = s_cum[E];

  // unit u -> expert e, panel m, token tiles [nt0, nt1) of width tw (the expert's rows spread
  // evenly over ceil(count / BN) tiles, rounded up to 16)
  struct Unit {
    int e, m, nt0, nt1, tw, cnt;
  };
  auto decode = [&](int u) {
    Unit d;
    d.e = find_expert(s_cum, E, u);
    d.cnt = s_off[d.e + 1] - s_off[d.e];
    const int ntiles = (d.cnt + Ws::BN - 1) / Ws::BN;
    d.tw = min(Ws::BN, ((d.cnt + ntiles - 1) / ntiles + 15) / 16 * 16);
    const int local = u - s_cum[d.e];
    d.m = local % p.MT;
    const int rb = local / p.MT;
    d.nt0 = rb * Ws::kTilesPerUnit;
    d.nt1 = min(ntiles, d.nt0 + Ws::kTilesPerUnit);
    return d;
  };

  if (warp == 0) {
    // ===================== weight panel, once per unit =====================
    if (lane == 0) {
      uint32_t a_phase = 0;
      const uint32_t tile_bytes = p.a_fp8 ? 2 * kTileCodeBytes : kTileCodeBytes;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit d = decode(u);
        // K-chunk kc of the panel is replaced as soon as the previous unit's last MMAs on it are done
        const int tile0 = (d.e * p.MT + d.m) * KC;
        bool okw = true;
        for (int kc = 0; kc < KC && okw; ++kc) {
          okw = mbar_wait(&a_empty[kc], a_phase ^ 1, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_EMPTY);
          if (!okw) break;
          mbar_arrive_expect_tx(&a_full[kc], tile_bytes + kTileScaleBytes);
          tma_load_2d(resA + kc * Ws::kTileA, &tmap_a, 0, (tile0 + kc) * 128, &a_full[kc]);
          bulk_load(resSfa + kc * 512, p.a_scales + (size_t)(tile0 + kc) * kTileScaleBytes, kTileScaleBytes,
                    &a_full[kc]);
        }
        if (!okw) break;
        a_phase ^= 1;
      }
    }
  } else if (warp == 1) {
    // ===================== token boxes and their scale bytes =====================
    // The chunks stream in order (units u, their token tiles nt, K-chunks kc). A chunk's scale
    // words are loaded one chunk ahead, before the previous chunk's are stored, so their latency
    // overlaps a whole chunk instead of stalling the stores.
    constexpr int NA = (Ws::BN + 127) / 128;
    int u = blockIdx.x, nt = 0, kn = 0;
    Unit d{};
    if (u < total) {
      d = decode(u);
      nt = d.nt0;
    }
    auto next_chunk = [&](int& row0, int& nrows, int& kc) {     // the chunk at the cursor, then advance
      if (u >= total) return false;
      row0 = s_off[d.e] + nt * d.tw;
      nrows = min(d.tw, d.cnt - nt * d.tw);
      kc = kn;
      if (++kn == KC) {
        kn = 0;
        if (++nt == d.nt1) {
          u += gridDim.x;
          if (u < total) {
            d = decode(u);
            nt = d.nt0;
          }
        }
      }
      return true;
    };
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int row0 = 0, nrows = 0, kc = 0;
    bool have = next_chunk(row0, nrows, kc);
    ScaleLines<NA> sl;
    if (have) load_scale_lines(sl, p.bs, p.b_scale_pitch, row0, nrows, kc, lane);
    while (have) {
      int row1 = 0, nrows1 = 0, kc1 = 0;
      const bool have1 = next_chunk(row1, nrows1, kc1);
      ScaleLines<NA> sl1;
      if (have1) load_scale_lines(sl1, p.bs, p.b_scale_pitch, row1, nrows1, kc1, lane);
      if (ok) ok = warp_wait(&empty[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_EMPTY);
      if (ok) {
        uint8_t* sB = stages + stage * Ws::kStageBytes;
        uint8_t* sSFB = sB + Ws::kTileB;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], Ws::kTileB);
          tma_load_2d(sB, &tmap_b, kc * 128, row0, &full[stage]);
        }
        store_scale_lines(sl, sSFB, lane);
        fence_async_smem();
        mbar_arrive(&full[stage]);
      }
      if (++stage == S) { stage = 0; phase ^= 1; }
      have = have1;
      row0 = row1;
      nrows = nrows1;
      kc = kc1;
      sl = sl1;
    }
  } else if (warp == 2) {
    // ===================== MMA issuer =====================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, a_phase = 0;
      int it = 0;
      bool ok = true;
      const uint32_t tsfa0 = tmem + Ws::kSfaCol;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit d = decode(u);
        for (int nt = d.nt0; nt < d.nt1 && ok; ++nt, ++it) {
          const bool first_tile = nt == d.nt0, last_tile = nt + 1 == d.nt1;
          const int tw = d.tw;
          const uint32_t idesc_base = idesc_mxf8f6f4(p.a_fp8 ? 0 : 5 /*weights E4M3 or E2M1*/, 0 /*E4M3*/, 128, tw, 0, 0);
          const int acc = it & 1;
          const int use = it >> 1;
          if (use > 0 &&
              !mbar_wait(&acc_empty[acc], (use - 1) & 1, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_DRAIN)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + (uint32_t)(acc * Ws::kAccStride);
          for (int kc = 0; kc < KC; ++kc) {
            if (first_tile) {
              // the unit's K-chunk kc of the panel has landed: its A scales go to their TMEM columns
              // (issued after the previous unit's MMAs that read them, in the tcgen05 pipe's order)
              if (!mbar_wait(&a_full[kc], a_phase, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_FULL)) {
                ok = false;
                break;
              }
              tc_fence_after();
              tc_cp_32x128b_warpx4(tsfa0 + 4 * kc, smem_desc(smem_u32(resSfa + kc * 512), 16, 128, 0));
            }
            if (!mbar_wait(&full[stage], phase, kWaitLimitNs, abort_flag, p.status, DEV_TIMEOUT_FULL)) {
              ok = false;
              break;
            }
            // (the token producer fenced its scale stores to the async proxy before arriving)
            tc_fence_after();
            uint8_t* sB = stages + stage * Ws::kStageBytes;
            uint8_t* sSFB = sB + Ws::kTileB;
            const uint32_t tsfb = tmem + Ws::kSfbCol + stage * Ws::kSfbSlot;
            for (int a = 0; a * 128 < tw; ++a)
              tc_cp_32x128b_warpx4(tsfb + 4 * a, smem_desc(smem_u32(sSFB + a * 512), 16, 128, 0));
            const uint32_t a0 = smem_u32(resA + kc * Ws::kTileA), b0 = smem_u32(sB);
            const int nk = min(4, (p.K - kc * 128) / 32);
            for (int kb = 0; kb < nk; ++kb) {
              const uint64_t ad = smem_desc(a0 + kb * 32, 16, 1024, 2);
              const uint64_t bd = smem_desc(b0 + kb * 32, 16, 1024, 2);
              const uint32_t id = idesc_base | ((uint32_t)kb << 4) | ((uint32_t)kb << 29);
              mma_mxf8f6f4(d_tmem, ad, bd, id, tsfa0 + 4 * kc, tsfb, (kc > 0 || kb > 0) ? 1u : 0u);
            }
            tc_commit(&empty[stage]);
            // after the unit's last MMAs on K-chunk kc, that chunk of the panel (and its TMEM scales)
            // may be replaced by the next unit's
            if (last_tile) tc_commit(&a_empty[kc]);
            if (++stage == S) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          tc_commit(&acc_full[acc]);
        }
        if (!ok) break;
        a_phase ^= 1;
      }
      tc_commit(drain);
      mbar_wait(drain, 0, kWaitLimitNs, nullptr, p.status, DEV_TIMEOUT_DRAIN);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ===================== epilogue (warp w -> TMEM lanes 32 (w % 4)) =====================
    const int qd = (warp - 4) & 3;
    const int half = (warp - 4) >> 2;
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    int it = 0;
    bool ok = true;
    constexpr int kGrp = 4;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit d = decode(u);
      for (int nt = d.nt0; nt < d.nt1; ++nt, ++it) {
        const int row0 = s_off[d.e] + nt * d.tw;
        const int nrows = min(d.tw, d.cnt - nt * d.tw);
        const int acc = it & 1;
        const int use = it >> 1;
        if (ok) ok = warp_wait(&acc_full[acc], use & 1, abort_flag, p.status, DEV_TIMEOUT_ACCUM);
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * Ws::kAccStride);
        for (int cg = 16 * kGrp * half; cg < d.tw; cg += 16 * kGrp * 2) {
          uint32_t rg[kGrp][16];
          if (ok) {
#pragma unroll
            for (int h = 0; h < kGrp; ++h)
              if (cg + 16 * h < d.tw) tmem_ld16(d_tmem + lane_base + cg + 16 * h, rg[h]);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < kGrp; ++h) reg_fence16(rg[h]);
#pragma unroll
            for (int h = 0; h < kGrp; ++h) {
              const int c0 = cg + 16 * h;
              if (c0 < d.tw) epi_w2_chunk<true>(rg[h], qd, lane, c0, d.m, row0, nrows, p);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(&acc_empty[acc]);
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
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, Ws::kTmemCols);
}

bool ws_down_supported(const moe_shape* s) {
  const int KC = ceil_div(s->I, kTileK);
  return KC <= Ws::kKcMax && (double)s->T * s->k / s->E > 64;
}

int launch_gemm_ws(const moe_shape* s, const uint8_t* codes, const GemmParams& gp, cudaStream_t st) {
  const long long slots = (long long)s->T * s->k;
  if (gp.KC > Ws::kKcMax) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)s->E * gp.MT * gp.KC * 128 >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap tm, tmb;
  const long long tiles = (long long)s->E * gp.MT * gp.KC;
  int rc = gp.a_fp8 ? make_weight_tmap_fp8(&tm, codes, tiles, 1) : make_weight_tmap(&tm, codes, tiles, 1);
  if (rc) return rc;
  rc = make_act_tmap(&tmb, gp.bq, gp.b_row_bytes, slots, Ws::BN);
  if (rc) return rc;
  if (ensure_smem_limit((const void*)grouped_gemm_ws_kernel, Ws::total(kMaxE))) return MOE_ERR_CUDA;
  // upper bound of the units: every expert's token tiles in blocks, times the panels
  const long long tiles_max = (slots + Ws::BN - 1) / Ws::BN + std::min<long long>(s->E, slots);
  const long long max_units = (long long)gp.MT * ((tiles_max + Ws::kTilesPerUnit - 1) / Ws::kTilesPerUnit +
                                                   std::min<long long>(s->E, slots));
  const long long grid = std::min<long long>(max_units, (long long)num_sms());
  if (grid <= 0) return MOE_OK;
  return launch_pdl(grouped_gemm_ws_kernel, dim3((unsigned)grid), dim3(Ws::kThreads), (size_t)Ws::total(gp.E), st, tm,
                    tmb, gp);
}

}  // namespace moe
