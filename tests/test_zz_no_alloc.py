"""The allocation-free router entry point (moe_route_topk_noalloc).

It exists for callers that cannot allocate device memory -- an engine that gave all of HBM to its
own pool at start-up, or code inside a host framework's callback where allocating is not allowed.
Its results must equal the workspace-based moe_route_topk bit for bit (routing is tested bit-exact
everywhere in this suite), on consecutive calls that share the library's internal scratch array.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def _inputs(T, H, E, seed, dead_frac=0.0):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((T, H)))
    wr = _bf16(rng.standard_normal((E, H)) * 0.02)
    bias = torch.from_numpy((rng.standard_normal(E) * 0.1).astype(np.float32)).cuda()
    dead = torch.from_numpy((rng.random(T) < dead_frac).astype(np.uint8)).cuda() if dead_frac else None
    return x, wr, bias, dead


def _same(a, b, S, Tk):
    assert torch.equal(a.topk_idx, b.topk_idx)
    assert torch.equal(a.topk_w.view(torch.int32), b.topk_w.view(torch.int32))
    assert torch.equal(a.expert_counts, b.expert_counts)
    assert torch.equal(a.expert_offsets, b.expert_offsets)
    assert torch.equal(a.slot_of_row[:S], b.slot_of_row[:S])
    assert torch.equal(a.row_of_slot[:Tk], b.row_of_slot[:Tk])


@pytest.mark.gpu
def test_noalloc_router_matches_workspace_router_on_consecutive_calls():
    from block_scaled_fp8_moe_gb300 import binding as B
    # a larger call first, then smaller ones with dead rows: a later call must not see an earlier
    # one's leftovers in the shared scratch. The three sizes cover each pair of router kernels the
    # two entry points pick (workspace / no-allocation): T = 200 screen + exact recompute / tiled,
    # T = 6 decode / small, T = 40 decode / tiled.
    for (T, H, E, k, seed, dead_frac) in ((200, 512, 256, 8, 1, 0.0), (6, 4096, 256, 8, 2, 0.3),
                                          (40, 4096, 256, 8, 3, 0.2)):
        x, wr, bias, dead = _inputs(T, H, E, seed, dead_frac)
        shp = B.shape(T, H, E, k, 64)
        ws = B.alloc_workspace(shp)
        ref = B.moe_route_topk(shp, x, wr, bias, dead, ws)
        got = B.moe_route_topk_noalloc(shp, x, wr, bias, dead)
        torch.cuda.synchronize()
        S = int(ref.expert_offsets[-1].item())
        _same(got, ref, S, T * k)


@pytest.mark.gpu
def test_noalloc_router_rejects_sizes_beyond_its_scratch():
    from block_scaled_fp8_moe_gb300 import binding as B
    n = ctypes.c_void_p(0)
    for (T, E) in ((257, 8), (128, 1024)):          # T > 256, T * E > 65536
        shp = B.shape(T, 256, E, 2, 64)
        rc = B.lib.moe_route_topk_noalloc(ctypes.byref(shp), *([n] * 10), n)
        assert rc == B.MOE_ERR_UNSUPPORTED_SHAPE
