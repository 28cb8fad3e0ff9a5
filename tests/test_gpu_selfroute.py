"""The layer call for a batch of at most 12 self-routed rows (no shared expert) runs the router and
then one GEMM launch that selects the top-k and builds the plan in each CTA (a warp takes one or two
rows). It must give the bits of the step entry points (route -> quant -> W13 -> W2 + combine), hand
the caller the same plan, and agree with the oracle; rows keep their bits across the 12 / 13 row
boundary, where the layer goes back to the separate plan kernel."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_moe_gb300 import synth
from tests import moe_harness as H

pytestmark = pytest.mark.gpu

CASES = [
    # name,    T,   H,   E,  k,   I, dead rows
    ("s1", 1, 256, 8, 2, 128, ()),
    ("s5", 5, 512, 64, 8, 192, (2,)),
    ("s8", 8, 256, 256, 8, 128, (0, 7)),
    ("s7e200", 7, 384, 200, 4, 256, ()),          # E not a multiple of 32
    ("s8k32", 8, 256, 64, 32, 128, (3,)),         # 256 slots, 32 choices per row
    ("s3e33", 3, 256, 33, 1, 64, ()),             # one choice per row
    ("s12", 12, 512, 64, 8, 192, (1, 11)),         # warps 0-3 select two rows each
    ("s10k32", 10, 256, 64, 32, 128, (9,)),       # 320 slots, two rows on warps 0 and 1
]


def _inter(T, k, E, Hd, I, dev, B):
    return dict(topk_idx=torch.full((T, k), -7, dtype=torch.int32, device=dev),
                topk_w=torch.full((T, k), float("nan"), dtype=torch.float32, device=dev),
                expert_counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
                expert_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                xq=torch.empty(T, Hd, dtype=torch.uint8, device=dev),
                xs=torch.empty(T, Hd // 32, dtype=torch.uint8, device=dev),
                hq=torch.empty(T * k, I, dtype=torch.uint8, device=dev),
                hs=torch.empty(T * k, B.hs_pitch(I), dtype=torch.uint8, device=dev))


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_self_routed_layer_equals_steps_and_oracle(case):
    name, T, Hd, E, k, I, dead_rows = case
    inp = synth.make_inputs_cpu(synth.custom(name, T, Hd, E, k, I, seed=11 * T + E))
    inp.dead[:] = 0
    for t in dead_rows:
        inp.dead[t] = 1
    g = H.GpuLayer(inp)
    B = g.B
    inter = _inter(T, k, E, Hd, I, g.x.device, B)
    dead = g.dead if dead_rows else None
    out = g.forward(dead=dead, inter=inter)
    B.moe_check_device_status(g.layer.workspace(T))
    st = g.run_steps(use_dead=bool(dead_rows))
    plan = st["plan"]
    torch.cuda.synchronize()
    # the plan handed to the caller is the plan kernel's
    assert torch.equal(inter["topk_idx"], plan.topk_idx)
    assert torch.equal(inter["topk_w"], plan.topk_w)
    assert torch.equal(inter["expert_counts"], plan.expert_counts)
    assert torch.equal(inter["expert_offsets"], plan.expert_offsets)
    S = int(plan.expert_offsets[-1].item())
    assert S == (T - len(dead_rows)) * k
    # same activation codes, same plan-order h rows, same output bits
    assert torch.equal(inter["xq"], st["xq"]) and torch.equal(inter["xs"], st["xs"])
    assert torch.equal(inter["hq"][:S], st["hq"][:S])
    assert torch.equal(inter["hs"][:S, : I // 32], st["hs"][:S, : I // 32])
    assert torch.equal(out, st["out"])
    # and the oracle
    ref, _, _ = H.oracle_forward(inp, use_dead=bool(dead_rows))
    assert np.array_equal(inter["topk_idx"].cpu().numpy(), ref.routing.topk_idx)
    assert np.array_equal(inter["topk_w"].cpu().numpy(), ref.routing.topk_w)
    got = H.bf16_to_np(out)
    H.assert_out_close(got, ref.out_exact)
    if dead_rows:
        d = np.array(dead_rows)
        assert np.all(got[d] == 0.0) and not np.any(np.signbit(got[d]))


def test_rows_keep_their_bits_across_the_twelve_row_boundary():
    inp = synth.make_inputs_cpu(synth.custom("b13", 13, 512, 64, 8, 192, seed=5))
    g = H.GpuLayer(inp)
    full = g.forward()                                     # plan kernel + one-launch GEMMs
    twelve = g.forward(x=g.x[:12].contiguous())            # routes itself
    nine = g.forward(x=g.x[3:12].contiguous())
    one = g.forward(x=g.x[12:13].contiguous())
    assert torch.equal(twelve, full[:12]) and torch.equal(nine, full[3:12]) and torch.equal(one[0], full[12])
    for t in (0, 7, 11):
        assert torch.equal(g.forward(x=g.x[t:t + 1].contiguous())[0], full[t])


def test_one_expert_pair_takes_every_row_and_all_dead():
    inp = synth.make_inputs_cpu(synth.custom("skew", 8, 256, 32, 2, 128, seed=3))
    inp.bias[:] = 0.0
    inp.bias[31] = 50.0
    inp.bias[4] = 40.0                                     # every row picks experts 31 and 4
    g = H.GpuLayer(inp)
    inter = _inter(8, 2, 32, 256, 128, g.x.device, g.B)
    out = g.forward(inter=inter)
    counts = inter["expert_counts"].cpu().numpy()
    assert counts[31] == 8 and counts[4] == 8 and counts.sum() == 16
    assert np.array_equal(inter["expert_offsets"].cpu().numpy()[[4, 5, 31, 32]], [0, 8, 8, 16])
    ref, _, _ = H.oracle_forward(inp, use_dead=False)
    H.assert_out_close(H.bf16_to_np(out), ref.out_exact)
    all_dead = g.forward(dead=torch.ones(8, dtype=torch.uint8, device="cuda"), inter=inter)
    assert torch.all(all_dead == 0) and not torch.any(torch.signbit(all_dead.float()))
    assert int(inter["expert_offsets"][-1].item()) == 0


def test_repeated_calls_alternating_with_the_plan_kernel_path():
    """Both paths share the GEMM's tile counters: each call's first kernel zeroes them."""
    inp = synth.make_inputs_cpu(synth.custom("alt", 40, 256, 64, 4, 128, seed=9))
    g = H.GpuLayer(inp)
    small = g.x[:6].contiguous()
    a = g.forward(x=small).clone()
    b = g.forward().clone()
    for _ in range(10):
        assert torch.equal(g.forward(x=small), a)
        assert torch.equal(g.forward(), b)
    assert torch.equal(a, b[:6])


def test_self_routed_layer_replays_from_a_cuda_graph():
    """The router inside the captured graph zeroes the GEMM's tile counters before every replay, and
    new rows copied into the captured input route afresh."""
    inp = synth.make_inputs_cpu(synth.custom("g6", 6, 512, 64, 8, 192, seed=21))
    g = H.GpuLayer(inp)
    other = synth.make_inputs_cpu(synth.custom("g6b", 6, 512, 64, 8, 192, seed=22))
    x2 = other.x.cuda()
    ref1 = g.forward().clone()
    ref2 = g.forward(x=x2).clone()
    xin = g.x.clone()
    out = torch.empty(6, 512, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.layer.forward(xin, out=out)                                    # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.layer.forward(xin, out=out)
    for _ in range(3):
        for x_new, ref in ((g.x, ref1), (x2, ref2)):
            xin.copy_(x_new)
            out.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, ref)
