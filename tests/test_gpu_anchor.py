"""GPU parity of anchored verify rows (TP4 serving profile README, settings table row "Verify
length"): a row with an anchor takes the anchor row's experts and weights them with its own
scores. Routing and plan bit-exact against the oracle (one-block and grid-wide plans, with dead
rows), the touched-expert set never grows, whole-layer output within tolerance, and invalid
anchors are ignored and reported."""
import numpy as np
import pytest
import torch

from oracle import moe as M
from tests import moe_harness as H

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _anchors(T, seed, frac=0.4):
    rng = np.random.default_rng(seed)
    anchor = np.full(T, -1, dtype=np.int32)
    n_self = max(1, T // 4)
    rows = rng.permutation(T)
    selfs, others = rows[:n_self], rows[n_self:]
    pick = others[rng.random(len(others)) < frac]
    anchor[pick] = rng.choice(selfs, size=len(pick))
    return anchor


@pytest.mark.parametrize("T,Hd,E,k", [(6, 4096, 256, 8), (37, 512, 16, 4), (300, 384, 32, 3), (700, 256, 64, 8)])
def test_anchored_routing_bit_exact(T, Hd, E, k):
    from block_scaled_fp8_moe_gb300 import binding as B
    rng = np.random.default_rng(T + E)
    x = _bf16(rng.standard_normal((T, Hd)))
    wr = _bf16(rng.standard_normal((E, Hd)) * 0.02)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    dead = (rng.random(T) < 0.2).astype(np.uint8)
    anchor = _anchors(T, seed=T)
    shp = B.shape(T, Hd, E, k, 64)
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, x.cuda(), wr.cuda(), torch.from_numpy(bias).cuda(), torch.from_numpy(dead).cuda(),
                            ws, anchor=torch.from_numpy(anchor).cuda())
    B.moe_check_device_status(ws)
    ref = M.route(x.float().numpy(), wr.float().numpy(), bias, k, dead.astype(bool), anchor)
    assert np.array_equal(plan.topk_idx.cpu().numpy(), ref.topk_idx)
    assert np.array_equal(plan.topk_w.cpu().numpy().view(np.uint32), ref.topk_w.view(np.uint32))
    assert np.array_equal(plan.expert_counts.cpu().numpy(), ref.counts)
    S = int(ref.offsets[-1])
    assert np.array_equal(plan.slot_of_row.cpu().numpy()[:S], ref.slot_of_row)
    assert np.array_equal(plan.row_of_slot.cpu().numpy()[:T * k], ref.row_of_slot)
    # the experts the batch touches are those its self-routed rows reach
    selfs = anchor < 0
    reached = set(ref.topk_idx[selfs].ravel().tolist())
    touched = set(np.nonzero(plan.expert_counts.cpu().numpy())[0].tolist())
    assert touched <= reached


def test_anchored_forward_matches_oracle():
    from block_scaled_fp8_moe_gb300 import synth
    inp = synth.make_inputs_cpu(synth.custom("anch37", 37, 512, 16, 4, 192, seed=41))
    g = H.GpuLayer(inp)
    anchor = _anchors(37, seed=3)
    out = g.forward(anchor=torch.from_numpy(anchor).cuda())
    ref, _, _ = H.oracle_forward(inp, anchor=anchor)
    H.assert_out_close(H.bf16_to_np(out), ref.out_exact)
    # self-routed rows give exactly the result of a batch without anchors
    plain = g.forward()
    same = np.nonzero(anchor < 0)[0]
    assert torch.equal(out[torch.from_numpy(same).cuda()], plain[torch.from_numpy(same).cuda()])


def test_invalid_anchors_are_ignored_and_reported():
    from block_scaled_fp8_moe_gb300 import binding as B
    T, Hd, E, k = 20, 256, 16, 4
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((T, Hd)))
    wr = _bf16(rng.standard_normal((E, Hd)) * 0.02)
    bias = np.zeros(E, np.float32)
    anchor = np.full(T, -1, dtype=np.int32)
    anchor[3] = 99          # out of range
    anchor[4], anchor[5] = 6, 4   # 5 points at an anchored row
    shp = B.shape(T, Hd, E, k, 64)
    ws = B.alloc_workspace(shp)
    plan = B.moe_route_topk(shp, x.cuda(), wr.cuda(), torch.from_numpy(bias).cuda(), None, ws,
                            anchor=torch.from_numpy(anchor).cuda())
    with pytest.raises(B.MoeError) as ei:
        B.moe_check_device_status(ws)
    assert ei.value.code == B.MOE_ERR_DEVICE_INPUT      # an input error, not an expired wait
    B.moe_check_device_status(ws)                      # the word was cleared
    fixed = anchor.copy()
    fixed[[3, 5]] = -1
    ref = M.route(x.float().numpy(), wr.float().numpy(), bias, k, None, fixed)
    assert np.array_equal(plan.topk_idx.cpu().numpy(), ref.topk_idx)
    assert np.array_equal(plan.topk_w.cpu().numpy(), ref.topk_w)
