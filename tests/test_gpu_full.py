"""Full-size workloads on the GPU, in the launch configuration bench.py times: sampled rows against
the oracle (routing and quantisation bit-exact, SwiGLU within 1e-5, output within 2e-2 x RMS,
weight codes bit-exact for the experts the samples reach) and batch invariance of whole rows."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_moe_gb300 import synth
from oracle import moe as M
from tests import moe_harness as Hh

pytestmark = pytest.mark.gpu

SAMPLES = {"decode-6": [0, 5], "decode-48": [3, 47], "prefill-4k": [7, 4095], "prefill-32k": [1, 30000]}


@pytest.fixture(scope="module")
def layers():
    from block_scaled_fp8_moe_gb300 import binding as B
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cfg = synth.CONFIGS[name]
            inp = synth.make_inputs_cuda(cfg)
            layer = B.MoeLayer.from_fp32(inp.w_router, inp.bias, inp.w13, inp.w2, cfg.k)
            cache[name] = (cfg, inp, layer)
        return cache[name]
    yield get
    cache.clear()
    torch.cuda.empty_cache()


def _run_full(B, cfg, inp, layer):
    T, k, I, H = cfg.T, cfg.k, cfg.I, cfg.H
    dev = inp.x.device
    inter = dict(topk_idx=torch.empty(T, k, dtype=torch.int32, device=dev),
                 topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
                 xq=torch.empty(T, H, dtype=torch.uint8, device=dev),
                 xs=torch.empty(T, H // 32, dtype=torch.uint8, device=dev),
                 hq=torch.empty(T * k, I, dtype=torch.uint8, device=dev),
                 hs=torch.empty(T * k, B.hs_pitch(I), dtype=torch.uint8, device=dev),
                 swiglu=torch.empty(T * k, I, dtype=torch.float32, device=dev))
    dead = inp.dead if cfg.dead_frac > 0 else None
    out = layer.forward(inp.x, dead=dead, inter=inter)
    B.moe_check_device_status(layer.workspace(T))
    # the plan row of every slot (the forward keeps it in its workspace): recompute with the router
    shp = layer.shape(T)
    plan = B.moe_route_topk(shp, inp.x, layer.w_router, layer.bias, dead, B.alloc_workspace(shp))
    torch.cuda.synchronize()
    assert torch.equal(plan.topk_idx, inter["topk_idx"])
    return out, inter, plan


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_sampled_rows_match_oracle(layers, name):
    from block_scaled_fp8_moe_gb300 import binding as B
    cfg, inp, layer = layers(name)
    out, inter, plan = _run_full(B, cfg, inp, layer)
    rows = SAMPLES[name]
    k = cfg.k
    x = inp.x[rows].float().cpu().numpy()
    wr = inp.w_router.float().cpu().numpy()
    bias = inp.bias.cpu().numpy()
    ro = M.route(x, wr, bias, k)
    # routing, bit-exact
    assert np.array_equal(inter["topk_idx"][rows].cpu().numpy(), ro.topk_idx)
    assert np.array_equal(inter["topk_w"][rows].cpu().numpy(), ro.topk_w)
    # activation quantisation, bit-exact
    rq, rs = M.quant_mxfp8(x)
    assert np.array_equal(inter["xq"][rows].cpu().numpy(), rq)
    assert np.array_equal(inter["xs"][rows].cpu().numpy(), rs)
    # weights the samples reach: the library's MXFP4 codes equal the oracle's
    used = sorted(set(ro.topk_idx.reshape(-1).tolist()))
    w13 = Hh.oracle_weights(inp.w13, used)
    w2 = Hh.oracle_weights(inp.w2, used)
    g13q, g13s = B.moe_quant_mxfp4(inp.w13[used[0]].contiguous())
    assert np.array_equal(g13q.cpu().numpy(), w13.codes[used[0]])
    assert np.array_equal(g13s.cpu().numpy(), w13.scales[used[0]])
    g2q, g2s = B.moe_quant_mxfp4(inp.w2[used[-1]].contiguous())
    assert np.array_equal(g2q.cpu().numpy(), w2.codes[used[-1]])
    assert np.array_equal(g2s.cpu().numpy(), w2.scales[used[-1]])
    # the sampled rows as their own batch (the oracle is row-independent)
    dead = inp.dead[rows].cpu().numpy().astype(bool) if cfg.dead_frac > 0 else None
    ref = M.forward(x, wr, bias, k, w13, w2, cfg.I, dead=dead)
    ros = plan.row_of_slot.cpu().numpy()
    for i, t in enumerate(rows):
        if dead is not None and dead[i]:
            assert torch.all(out[t] == 0)
            continue
        for j in range(k):
            pg = ros[t * k + j]
            po = ref.routing.row_of_slot[i * k + j]
            n = int(np.nonzero(ref.w13.rows == po)[0][0])
            a_ref = ref.w13.a[n]
            a_gpu = inter["swiglu"][pg].double().cpu().numpy()
            rms = np.sqrt(np.mean(a_ref ** 2))
            assert np.all(np.abs(a_gpu - a_ref) <= Hh.SWIGLU_REL * np.maximum(np.abs(a_ref), rms))
            gq = inter["hq"][pg].cpu().numpy()[None]
            gs = inter["hs"][pg].cpu().numpy()[None]
            bq, bs = Hh.e4m3_codes_match(gq, gs, ref.w13.hq[n][None], ref.w13.hs[n][None], ref.w13.flip_ok[n][None])
            assert bq == 0 and bs == 0
    live = [i for i in range(len(rows)) if dead is None or not dead[i]]
    Hh.assert_out_close(out[rows].float().cpu().numpy()[live], ref.out_exact[live])


@pytest.mark.parametrize("name,subsets", [
    ("decode-6", [(0, 1), (5, 6), (2, 5)]),
    ("prefill-4k", [(0, 6), (100, 148), (4095, 4096)]),
    ("prefill-32k", [(0, 6), (1000, 1048), (20000, 20256), (32767, 32768)]),
])
def test_full_size_batch_invariance(layers, name, subsets):
    cfg, inp, layer = layers(name)
    full = layer.forward(inp.x).clone()
    for lo, hi in subsets:
        part = layer.forward(inp.x[lo:hi].contiguous())
        assert torch.equal(part, full[lo:hi]), (lo, hi)


def test_decode48_rows_alone_and_dead_rows(layers):
    cfg, inp, layer = layers("decode-48")
    full = layer.forward(inp.x, dead=inp.dead).clone()
    dead = inp.dead.bool()
    assert int(dead.sum()) == 14
    assert torch.all(full[dead] == 0)
    for t in range(cfg.T):
        if dead[t]:
            continue
        one = layer.forward(inp.x[t:t + 1].contiguous())
        assert torch.equal(one[0], full[t]), t
