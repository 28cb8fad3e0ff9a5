"""Full-size workloads on the GPU, in the launch configuration bench.py times, against the oracle.

Whole batch: the routing (indices, weights), the plan (counts, offsets, slot lists) and the MXFP8
activation codes and scales of EVERY row are compared bit for bit ("New Deepseek 4.1 flash recipe",
post 4 "Quality and correctness": exact selections; post 6 "Why TileLang": fixed-order reductions).
The oracle's row-independent steps run over a pool of spawned processes (tests/oracle_pool.py).

Sampled from the plan: the pre-requant SwiGLU (within 1e-5) and requant codes of plan rows at the
first, last and middle token tiles of the three most-loaded experts (and of the least-loaded one),
for the tile widths the two GEMMs use at that size; the final output (within 2e-2 x RMS) of the
tokens those rows belong to plus the last row of the batch. Decode batches check every row.
Batch invariance of whole rows at full size is checked separately."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_moe_gb300 import synth
from oracle import moe as M
from tests import moe_harness as Hh
from tests import oracle_pool

pytestmark = pytest.mark.gpu

WIDE_BN = 224          # widest token tile of the prefill GEMMs
SHORT_K_CHUNKS = 8     # down projections with fewer K-chunks of 128 keep 128-row tiles


@pytest.fixture(scope="module")
def pool():
    with oracle_pool.Pool() as p:
        yield p


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
                 expert_counts=torch.empty(cfg.E, dtype=torch.int32, device=dev),
                 expert_offsets=torch.empty(cfg.E + 1, dtype=torch.int32, device=dev),
                 xq=torch.empty(T, H, dtype=torch.uint8, device=dev),
                 xs=torch.empty(T, H // 32, dtype=torch.uint8, device=dev),
                 hq=torch.empty(T * k, I, dtype=torch.uint8, device=dev),
                 hs=torch.empty(T * k, B.hs_pitch(I), dtype=torch.uint8, device=dev),
                 swiglu=torch.empty(T * k, I, dtype=torch.float32, device=dev))
    dead = inp.dead if cfg.dead_frac > 0 else None
    out = layer.forward(inp.x, dead=dead, inter=inter)
    B.moe_check_device_status(layer.workspace(T))
    # the slot lists stay in the forward's workspace: the router entry point writes them again
    shp = layer.shape(T)
    plan = B.moe_route_topk(shp, inp.x, layer.w_router, layer.bias, dead, B.alloc_workspace(shp))
    torch.cuda.synchronize()
    assert torch.equal(plan.topk_idx, inter["topk_idx"])
    assert torch.equal(plan.expert_offsets, inter["expert_offsets"])
    return out, inter, plan


def _tile_width(cfg, cnt, w13: bool):
    """Token-tile width (columns) the grouped GEMM gives an expert with `cnt` plan rows."""
    avg = cfg.T * cfg.k / cfg.E
    bn = 16 if avg <= 16 else 32 if avg <= 32 else 64 if avg <= 64 else WIDE_BN
    if not w13 and bn > 128 and -(-cfg.I // 128) < SHORT_K_CHUNKS:
        bn = 128
    if bn < WIDE_BN:
        return bn
    ntiles = -(-cnt // WIDE_BN)
    return min(WIDE_BN, (-(-cnt // ntiles) + 15) // 16 * 16)


def _tile_rows(cfg, offsets, e):
    """Plan rows at the first, middle and last column of the first, middle and last token tile of
    expert e, for the tile widths of both GEMMs."""
    lo, hi = int(offsets[e]), int(offsets[e + 1])
    cnt = hi - lo
    rows = set()
    for w13 in (True, False):
        tw = _tile_width(cfg, cnt, w13)
        starts = list(range(0, cnt, tw))
        for s in {starts[0], starts[len(starts) // 2], starts[-1]}:
            end = min(s + tw, cnt)
            rows.update((lo + s, lo + (s + end - 1) // 2, lo + end - 1))
    return sorted(rows)


@pytest.mark.parametrize("name", ["decode-6", "decode-48", "prefill-4k", "prefill-32k"])
def test_full_size_whole_batch_against_oracle(layers, pool, name):
    from block_scaled_fp8_moe_gb300 import binding as B
    cfg, inp, layer = layers(name)
    out, inter, plan = _run_full(B, cfg, inp, layer)
    T, k, E, I = cfg.T, cfg.k, cfg.E, cfg.I
    x = inp.x.float().cpu().numpy()
    wr = inp.w_router.float().cpu().numpy()
    bias = inp.bias.cpu().numpy()
    dead = inp.dead.cpu().numpy().astype(bool) if cfg.dead_frac > 0 else None

    # ---- every row: routing and plan bit-exact ----
    ro = pool.route_all(x, wr, bias, k, dead)
    S = int(ro.offsets[-1])
    assert np.array_equal(inter["topk_idx"].cpu().numpy(), ro.topk_idx)
    assert np.array_equal(inter["topk_w"].cpu().numpy().view(np.int32), ro.topk_w.view(np.int32))
    assert np.array_equal(inter["expert_counts"].cpu().numpy(), ro.counts)
    assert np.array_equal(plan.expert_offsets.cpu().numpy(), ro.offsets)
    assert np.array_equal(plan.slot_of_row.cpu().numpy()[:S], ro.slot_of_row)
    assert np.array_equal(plan.row_of_slot.cpu().numpy()[:T * k], ro.row_of_slot)

    # ---- every row: MXFP8 activation codes and scales bit-exact ----
    xq_o, xs_o = pool.quant_all(x)
    assert np.array_equal(inter["xq"].cpu().numpy(), xq_o)
    assert np.array_equal(inter["xs"].cpu().numpy(), xs_o)

    # ---- plan rows at tile boundaries of the heaviest experts (every row of a decode batch) ----
    if T <= 64:
        rows = np.arange(S)
    else:
        order = np.argsort(-ro.counts, kind="stable")
        picked = list(order[:3]) + [int(order[np.count_nonzero(ro.counts) - 1])]
        rows = np.array(sorted({r for e in picked for r in _tile_rows(cfg, ro.offsets, int(e))}))
    tokens = sorted({int(ro.slot_of_row[p]) // k for p in rows} | {T - 1})
    if T > 64:
        assert len(rows) >= 12
    # every expert the checked tokens reach, quantised by the oracle from the fp32 weights
    experts = sorted(set(ro.topk_idx[tokens].reshape(-1).tolist()) |
                     set(int(np.searchsorted(ro.offsets, p, side="right") - 1) for p in rows))
    w13 = pool.weights(lambda e: inp.w13[e].cpu().numpy(), E, 2 * I, cfg.H, experts)
    w2 = pool.weights(lambda e: inp.w2[e].cpu().numpy(), E, cfg.H, I, experts)

    r13 = M.w13_swiglu(xq_o, xs_o, w13, ro, k, I, rows)
    a_gpu = inter["swiglu"][torch.from_numpy(rows).to(inter["swiglu"].device)].double().cpu().numpy()
    rms = np.sqrt(np.mean(r13.a ** 2, axis=1, keepdims=True))
    tol = Hh.SWIGLU_REL * np.maximum(np.abs(r13.a), rms)
    assert np.all(np.abs(a_gpu - r13.a) <= tol), float(np.max(np.abs(a_gpu - r13.a) / tol))
    sel = torch.from_numpy(rows).to(inter["hq"].device)
    bq, bs = Hh.e4m3_codes_match(inter["hq"][sel].cpu().numpy(), inter["hs"][sel].cpu().numpy(), r13.hq, r13.hs,
                                 r13.flip_ok)
    assert bq == 0 and bs == 0

    # ---- output of the tokens those rows belong to (rows are independent in the oracle) ----
    tk = np.array(tokens)
    ref = M.forward(x[tk], wr, bias, k, w13, w2, I, dead=None if dead is None else dead[tk])
    got = out[torch.from_numpy(tk).to(out.device)].float().cpu().numpy()
    live = np.ones(len(tk), bool) if dead is None else ~dead[tk]
    assert np.all(got[~live] == 0)
    Hh.assert_out_close(got[live], ref.out_exact[live])


def test_full_size_weight_codes_match_oracle(layers, pool):
    """The library's MXFP4 weight codes equal the oracle's for a few experts at the full shape."""
    from block_scaled_fp8_moe_gb300 import binding as B
    cfg, inp, layer = layers("prefill-32k")
    for e in (0, cfg.E - 1):
        w = pool.weights(lambda i: inp.w13[i].cpu().numpy(), cfg.E, 2 * cfg.I, cfg.H, [e])
        gq, gs = B.moe_quant_mxfp4(inp.w13[e].contiguous())
        assert np.array_equal(gq.cpu().numpy(), w.codes[e])
        assert np.array_equal(gs.cpu().numpy(), w.scales[e])
        w = pool.weights(lambda i: inp.w2[i].cpu().numpy(), cfg.E, cfg.H, cfg.I, [e])
        gq, gs = B.moe_quant_mxfp4(inp.w2[e].contiguous())
        assert np.array_equal(gq.cpu().numpy(), w.codes[e])
        assert np.array_equal(gs.cpu().numpy(), w.scales[e])


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
