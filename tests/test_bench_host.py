"""Host-side checks of bench.py: the per-step launch count it reports (`gpu_launches`) follows the
library's dispatch, whose constants are read from the CUDA sources so that a change there that
is not mirrored here fails on the CPU."""
import os
import re

import bench
from block_scaled_fp8_moe_gb300 import synth

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "block_scaled_fp8_moe_gb300",
                    "csrc")


def _const(name, fname="route.cu"):
    src = open(os.path.join(CSRC, fname)).read()
    m = re.search(r"#define %s (\d+)" % name, src) or re.search(r"constexpr \w+ %s = ([\d *]+);" % name, src)
    assert m, name
    return eval(m.group(1))  # noqa: S307 - integer literals / products from our own source


def _decode_router(T, H, E=256):
    nc = H // 64
    small = T <= _const("kDecSmallT")
    ept = 1 if small else 2
    epc = min(E, _const("kDecEpcSmall") if small else _const("kDecEpcLarge"))
    tpc = min(T, _const("kDecTpcSmall")) if small else _const("kDecTpcLarge")
    pitch, cap = _const("kDecPitch"), _const("kDecodeSmemMax")

    def smem(tp):
        return tp * nc * pitch + epc * tp * (nc + 1) * 4

    while tpc > 1 and smem(tpc) > cap:
        tpc -= 1
    threads = -(-epc // ept) * nc
    return T <= _const("kDecMaxT") and threads <= _const("kDecThreadsMax") and smem(tpc) <= cap


def test_decode_router_predicate_matches_the_library_constants():
    for T in (1, 6, 10, 11, 12, 16, 48, 64, 65):
        for H in (256, 4096, 8192, 16384):
            cfg = synth.custom("p", T, H, 256, 8, 128, seed=0)
            n = bench.launches_per_step(cfg)
            fused = 2 if T * 8 / 256 <= 32 else 0          # one launch for W13 + W2 + combine (decode tiles)
            self_routed = T <= _const("kSelfPlanMaxT", "common.cuh") and _const("kSelfPlanMaxE", "common.cuh") >= 256
            if _decode_router(T, H) and self_routed:
                assert n == 2, (T, H)              # router (+ quant), GEMMs that route the rows themselves
            elif _decode_router(T, H):
                # router (+ quant), top-k + plan (a grid-wide top-k first above 24 rows), W13, W2, combine
                assert n == 5 - fused + (1 if T > 24 else 0), (T, H)
            else:
                assert n >= 6 - fused, (T, H)      # separate quantiser and a non-decode router


def test_launch_counts_of_the_benchmarked_workloads():
    counts = {name: bench.launches_per_step(synth.CONFIGS[name]) for name in
              ("decode-6", "decode-48", "prefill-4k", "prefill-32k")}
    # decode-6: fused router+quant, then top-k, plan, W13 + W2 + combine in one launch; decode-48:
    # the same with a grid-wide top-k and the one-CTA plan between them; prefill: norms, screen,
    # exact recompute, grid-wide select, plan, scan, scatter, quantiser into plan order, W13, W2,
    # combine
    assert counts == {"decode-6": 2, "decode-48": 4, "prefill-4k": 11, "prefill-32k": 11}
    # with a shared expert the combine is its own launch after the side stream joins
    assert bench.launches_per_step(synth.CONFIGS["decode-6"], shared=True) == 7


def test_gemm_kind_classifies_every_grouped_gemm_launch_name():
    """The traffic recorder files each ncu launch under the step it belongs to."""
    ck = "(CUtensorMap_st, CUtensorMap_st, CUtensorMap_st, GemmParams, GemmParams)"
    assert bench.gemm_kind("void grouped_gemm_kernel<16, 2>" + ck) == "experts"
    assert bench.gemm_kind("void grouped_gemm_kernel<16, 3>" + ck) == "experts_selfroute"
    assert bench.gemm_kind("void grouped_gemm_kernel<224, 1>" + ck) == "w13"
    assert bench.gemm_kind("void grouped_gemm_kernel<64, 0>" + ck) == "w2"
    assert bench.gemm_kind("grouped_gemm_ws_kernel(CUtensorMap_st, CUtensorMap_st, GemmParams)") == "w2"
    assert bench.gemm_kind("void grouped_gemm_pair_kernel<true, PairCfg<192, 3, 2>>(...)") == "w13"
    assert bench.gemm_kind("void grouped_gemm_pair_kernel<false, PairCfg<192, 3, 2>>(...)") == "w2"
    assert bench.gemm_kind("void combine_kernel(const float *, ...)") is None
    assert bench.gemm_kind("void quant_mxfp8_plan_kernel(...)") is None
