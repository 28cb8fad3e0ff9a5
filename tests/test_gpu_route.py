"""GPU parity: router logits / sigmoid / top-k / weights / plan, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from oracle import moe as M

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _route_case(T, H, E, k, seed, dead_frac=0.0, ties=False, bias_scale=0.1):
    from block_scaled_fp8_moe_gb300 import binding as B
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((T, H)))
    wr = _bf16(rng.standard_normal((E, H)) * 0.02)
    bias = (rng.standard_normal(E) * bias_scale).astype(np.float32)
    if ties:
        wr[E - 1] = wr[1]
        wr[E // 2] = wr[0]
        bias[E - 1] = bias[1]
        bias[E // 2] = bias[0]
    dead = (rng.random(T) < dead_frac).astype(np.uint8)
    shp = B.shape(T, H, E, k, 64)
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, x.cuda(), wr.cuda(), torch.from_numpy(bias).cuda(),
                            torch.from_numpy(dead).cuda() if dead_frac > 0 else None, ws)
    B.moe_check_device_status(ws)
    ref = M.route(x.float().numpy(), wr.float().numpy(), bias, k, dead.astype(bool) if dead_frac > 0 else None)
    return plan, ref


@pytest.mark.parametrize("T,H,E,k", [
    (1, 256, 8, 2), (4, 256, 8, 2), (6, 4096, 256, 8), (7, 512, 64, 6), (16, 256, 32, 4), (17, 256, 32, 4),
    (33, 384, 16, 3), (65, 128, 8, 8), (256, 256, 64, 8), (257, 256, 64, 8), (600, 512, 40, 5),
    (4, 8192, 32, 4), (11, 8192, 16, 2),      # decode router at its widest rows (128 chunks per row)
    (28, 1024, 256, 8), (48, 4096, 256, 8),   # grid-wide top-k, then the one-CTA plan from its lists
])
def test_route_bit_exact(T, H, E, k):
    plan, ref = _route_case(T, H, E, k, seed=T * 31 + E)
    assert np.array_equal(plan.topk_idx.cpu().numpy(), ref.topk_idx)
    assert np.array_equal(plan.topk_w.cpu().numpy().view(np.uint32), ref.topk_w.view(np.uint32))
    assert np.array_equal(plan.expert_counts.cpu().numpy(), ref.counts)
    assert np.array_equal(plan.expert_offsets.cpu().numpy(), ref.offsets)
    S = int(ref.offsets[-1])
    assert np.array_equal(plan.slot_of_row.cpu().numpy()[:S], ref.slot_of_row)
    assert np.array_equal(plan.row_of_slot.cpu().numpy()[:T * k], ref.row_of_slot)


@pytest.mark.parametrize("E,n_tied", [(64, 40), (128, 100)])
def test_route_screen_long_candidate_lists(E, n_tied):
    """Screened routing (T = 300) where every row's candidate list is long: n_tied experts share one
    router row and a bias that puts them on top, so each row has at least n_tied candidates (40: a
    long list; 100: more than a list holds, every expert recomputed). The tied keys are equal, so
    the lowest expert ids win."""
    from block_scaled_fp8_moe_gb300 import binding as B
    T, H, k = 300, 256, 8
    rng = np.random.default_rng(E + n_tied)
    x = _bf16(rng.standard_normal((T, H)))
    wr = _bf16(rng.standard_normal((E, H)) * 0.02)
    wr[:n_tied] = wr[0]
    bias = (rng.standard_normal(E) * 0.01).astype(np.float32)
    bias[:n_tied] = 1.0
    shp = B.shape(T, H, E, k, 64)
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, x.cuda(), wr.cuda(), torch.from_numpy(bias).cuda(), None, ws)
    B.moe_check_device_status(ws)
    ref = M.route(x.float().numpy(), wr.float().numpy(), bias, k, None)
    assert np.array_equal(ref.topk_idx, np.tile(np.arange(k, dtype=ref.topk_idx.dtype), (T, 1)))
    assert np.array_equal(plan.topk_idx.cpu().numpy(), ref.topk_idx)
    assert np.array_equal(plan.topk_w.cpu().numpy().view(np.uint32), ref.topk_w.view(np.uint32))
    assert np.array_equal(plan.expert_offsets.cpu().numpy(), ref.offsets)


@pytest.mark.parametrize("T", [5, 48, 300])
def test_route_dead_rows_and_ties(T):
    plan, ref = _route_case(T, 256, 16, 4, seed=T, dead_frac=0.3, ties=True)
    assert np.array_equal(plan.topk_idx.cpu().numpy(), ref.topk_idx)
    assert np.array_equal(plan.topk_w.cpu().numpy(), ref.topk_w)
    assert np.array_equal(plan.expert_offsets.cpu().numpy(), ref.offsets)
    S = int(ref.offsets[-1])
    assert np.array_equal(plan.slot_of_row.cpu().numpy()[:S], ref.slot_of_row)
    assert np.array_equal(plan.row_of_slot.cpu().numpy()[:T * 4], ref.row_of_slot)


def test_route_skewed_bias_all_slots_to_few_experts():
    plan, ref = _route_case(300, 256, 16, 2, seed=9, bias_scale=10.0)
    assert np.array_equal(plan.topk_idx.cpu().numpy(), ref.topk_idx)
    assert np.array_equal(plan.expert_counts.cpu().numpy(), ref.counts)
    assert (ref.counts == 0).sum() >= 10          # most experts empty


def _survival_edges(n, seed):
    rng = np.random.default_rng(seed)
    p = rng.random(n).astype(np.float32)
    p[:8] = [0.0, np.nextafter(np.float32(0.2), np.float32(0)), 0.2, np.nextafter(np.float32(0.2), np.float32(1)),
             np.nan, -np.inf, np.inf, -0.0]
    return p


def test_dead_from_survival_bit_exact():
    from block_scaled_fp8_moe_gb300 import binding as B
    for n, thr in ((1, 0.2), (8, 0.2), (1000, 0.2), (4097, 0.35)):
        p = _survival_edges(max(n, 8), n)[:n]
        d = B.moe_dead_from_survival(torch.from_numpy(p).cuda(), thr)
        torch.cuda.synchronize()
        assert np.array_equal(d.cpu().numpy(), M.dead_from_survival(p, thr))


def test_route_with_survival_mask_matches_oracle():
    from block_scaled_fp8_moe_gb300 import binding as B
    T, H, E, k = 37, 256, 16, 4
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((T, H)))
    wr = _bf16(rng.standard_normal((E, H)) * 0.02)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    p = _survival_edges(T, 9)
    dead = B.moe_dead_from_survival(torch.from_numpy(p).cuda())
    shp = B.shape(T, H, E, k, 64)
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, x.cuda(), wr.cuda(), torch.from_numpy(bias).cuda(), dead, ws)
    B.moe_check_device_status(ws)
    ref = M.route(x.float().numpy(), wr.float().numpy(), bias, k, M.dead_from_survival(p).astype(bool))
    S = int(ref.offsets[-1])
    assert np.array_equal(plan.expert_offsets.cpu().numpy(), ref.offsets)
    assert np.array_equal(plan.slot_of_row.cpu().numpy()[:S], ref.slot_of_row)
    assert np.array_equal(plan.row_of_slot.cpu().numpy(), ref.row_of_slot)
