"""The down projection and the combine as separate calls (moe_w2_grouped, moe_combine) give the same
bits as the fused moe_w2_combine_grouped, and the `dead` mask given to the combine forces +0.0 rows
and reports a plan that still gives a flagged row slots."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_moe_gb300 import synth
from tests import moe_harness as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T,Hd,E,k,I,dead_frac", [
    ("s37", 37, 512, 16, 4, 192, 0.25),      # decode-sized tiles, dead rows
    ("s640", 640, 256, 4, 2, 1024, 0.0),     # wide tiles in both GEMMs
])
def test_split_w2_and_combine_equal_fused(name, T, Hd, E, k, I, dead_frac):
    from block_scaled_fp8_moe_gb300 import binding as B
    inp = synth.make_inputs_cpu(synth.custom(name, T, Hd, E, k, I, seed=T + 7, dead_frac=dead_frac))
    g = H.GpuLayer(inp)
    shp = g.shape()
    ws = B.alloc_workspace(shp)
    dead = g.dead if dead_frac else None
    plan = B.moe_route_topk(shp, g.x, g.wr, g.bias, dead, ws)
    xq, xs = B.moe_quant_mxfp8(g.x)
    hq, hs = B.moe_w13_swiglu_grouped(shp, xq, xs, g.layer.w13p, g.layer.w13sp, plan, ws)
    fused = B.moe_w2_combine_grouped(shp, hq, hs, g.layer.w2p, g.layer.w2sp, plan, ws, dead=dead).clone()
    y = B.moe_w2_grouped(shp, hq, hs, g.layer.w2p, g.layer.w2sp, plan, ws)
    split = B.moe_combine(shp, y, plan, ws, dead=dead)
    B.moe_check_device_status(ws)
    assert torch.equal(split, fused)
    # and the whole layer agrees with both
    assert torch.equal(g.forward(dead=dead), fused)
    ref, _, _ = H.oracle_forward(inp, use_dead=dead is not None)
    H.assert_out_close(H.bf16_to_np(split), ref.out_exact)


def test_dead_mask_on_a_plan_made_without_it():
    from block_scaled_fp8_moe_gb300 import binding as B
    inp = synth.make_inputs_cpu(synth.custom("s20", 20, 256, 8, 2, 128, seed=9, dead_frac=0.3))
    g = H.GpuLayer(inp)
    shp = g.shape()
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, g.x, g.wr, g.bias, None, ws)          # every row holds slots
    xq, xs = B.moe_quant_mxfp8(g.x)
    hq, hs = B.moe_w13_swiglu_grouped(shp, xq, xs, g.layer.w13p, g.layer.w13sp, plan, ws)
    plain = B.moe_w2_combine_grouped(shp, hq, hs, g.layer.w2p, g.layer.w2sp, plan, ws).clone()
    B.moe_check_device_status(ws)
    masked = B.moe_w2_combine_grouped(shp, hq, hs, g.layer.w2p, g.layer.w2sp, plan, ws, dead=g.dead)
    with pytest.raises(B.MoeError) as ei:
        B.moe_check_device_status(ws)
    assert ei.value.code == B.MOE_ERR_DEVICE_INPUT
    flagged = g.dead.bool()
    assert int(flagged.sum()) == 6
    assert torch.all(masked[flagged] == 0) and not torch.any(torch.signbit(masked[flagged].float()))
    assert torch.equal(masked[~flagged], plain[~flagged])


@pytest.mark.parametrize("name,T,Hd,E,k,I", [("p37", 37, 512, 16, 4, 192), ("p640", 640, 256, 4, 2, 1024)])
def test_w13_on_plan_order_rows_equals_token_order(name, T, Hd, E, k, I):
    """moe_quant_mxfp8_plan + MOE_FLAG_X_PLAN_ORDER (what moe_forward runs for wide tiles) against
    token-order codes: plan rows are copies of their tokens' codes, and W13 gives the same bits."""
    from block_scaled_fp8_moe_gb300 import binding as B
    inp = synth.make_inputs_cpu(synth.custom(name, T, Hd, E, k, I, seed=T + 11, dead_frac=0.2))
    g = H.GpuLayer(inp)
    shp = g.shape()
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, g.x, g.wr, g.bias, g.dead, ws)
    xq, xs = B.moe_quant_mxfp8(g.x)
    xq2 = torch.empty_like(xq)
    xs2 = torch.empty_like(xs)
    xqp, xsp = B.moe_quant_mxfp8_plan(shp, g.x, plan, xq=xq2, xs=xs2)
    S = int(plan.expert_offsets[-1].item())
    tok = (plan.slot_of_row[:S] // k).long()
    assert torch.equal(xq2, xq) and torch.equal(xs2, xs)
    assert torch.equal(xqp[:S], xq[tok]) and torch.equal(xsp[:S], xs[tok])
    hq, hs = B.moe_w13_swiglu_grouped(shp, xq, xs, g.layer.w13p, g.layer.w13sp, plan, ws)
    shp_p = g.shape(flags=B.MOE_FLAG_X_PLAN_ORDER)
    hq2, hs2 = B.moe_w13_swiglu_grouped(shp_p, xqp, xsp, g.layer.w13p, g.layer.w13sp, plan, ws)
    B.moe_check_device_status(ws)
    assert torch.equal(hq[:S], hq2[:S])
    assert torch.equal(hs[:S, : I // 32], hs2[:S, : I // 32])
