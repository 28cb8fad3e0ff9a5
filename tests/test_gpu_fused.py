"""Both expert GEMMs through moe_experts_grouped (one persistent launch for decode-sized batches)
give the same bits as moe_w13_swiglu_grouped followed by moe_w2_grouped, on repeated calls (the
per-expert counters start from zero every call), with dead rows, and at the decode-6 shape."""
import pytest
import torch

from block_scaled_fp8_moe_gb300 import synth
from tests import moe_harness as H

pytestmark = pytest.mark.gpu


def _both(B, shp, xq, xs, layer, plan, ws):
    S = int(plan.expert_offsets[-1].item())
    hq, hs = B.moe_w13_swiglu_grouped(shp, xq, xs, layer.w13p, layer.w13sp, plan, ws)
    y = B.moe_w2_grouped(shp, hq, hs, layer.w2p, layer.w2sp, plan, ws)
    return hq[:S].clone(), hs[:S].clone(), y[:S].clone(), S


@pytest.mark.parametrize("name,T,Hd,E,k,I,dead_frac", [
    ("f37", 37, 512, 16, 4, 192, 0.25),     # 16-row tiles, 3 W13 panels
    ("f100", 100, 256, 8, 2, 256, 0.0),     # 32-row tiles
    ("f5", 5, 256, 8, 2, 576, 0.0),         # down projection with a partial last K-chunk
])
def test_experts_grouped_equals_two_gemms(name, T, Hd, E, k, I, dead_frac):
    from block_scaled_fp8_moe_gb300 import binding as B
    inp = synth.make_inputs_cpu(synth.custom(name, T, Hd, E, k, I, seed=T + 3, dead_frac=dead_frac))
    g = H.GpuLayer(inp)
    shp = g.shape()
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, g.x, g.wr, g.bias, g.dead if dead_frac else None, ws)
    xq, xs = B.moe_quant_mxfp8(g.x)
    hq, hs, y, S = _both(B, shp, xq, xs, g.layer, plan, ws)
    for _ in range(3):
        hq2, hs2, y2 = B.moe_experts_grouped(shp, xq, xs, g.layer.w13p, g.layer.w13sp, g.layer.w2p, g.layer.w2sp,
                                             plan, ws)
        B.moe_check_device_status(ws)
        assert torch.equal(hq2[:S], hq) and torch.equal(hs2[:S, : I // 32], hs[:, : I // 32])
        assert torch.equal(y2[:S], y)


def test_experts_grouped_at_decode6():
    from block_scaled_fp8_moe_gb300 import binding as B
    cfg = synth.CONFIGS["decode-6"]
    inp = synth.make_inputs_cuda(cfg)
    layer = B.MoeLayer.from_fp32(inp.w_router, inp.bias, inp.w13, inp.w2, cfg.k)
    del inp.w13, inp.w2
    shp = layer.shape(cfg.T)
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, inp.x, layer.w_router, layer.bias, None, ws)
    xq, xs = B.moe_quant_mxfp8(inp.x)
    hq, hs, y, S = _both(B, shp, xq, xs, layer, plan, ws)
    for _ in range(3):
        hq2, hs2, y2 = B.moe_experts_grouped(shp, xq, xs, layer.w13p, layer.w13sp, layer.w2p, layer.w2sp, plan, ws)
        B.moe_check_device_status(ws)
        assert torch.equal(hq2[:S], hq) and torch.equal(hs2[:S], hs) and torch.equal(y2[:S], y)
    # and the whole layer (the forward runs the same GEMMs) against the step entry points
    out = layer.forward(inp.x)
    ref = B.moe_combine(shp, y, plan, ws)
    assert torch.equal(out, ref)
