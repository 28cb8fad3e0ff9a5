"""GPU parity of the shared expert (TP4 serving profile README: a dense MXFP8 SwiGLU expert on a
side stream beside the routed ones, added after the routed slots): whole-layer output against
the oracle at narrow and wide token tiles with dead rows, side stream and same stream identical,
zero shared weights identical to no shared expert, and batch invariance of whole rows."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_moe_gb300 import synth
from oracle import formats as F
from oracle import moe as M
from tests import moe_harness as H

pytestmark = pytest.mark.gpu


def _shared_codes(Hd, Is, seed, zero=False):
    rng = np.random.default_rng(seed)
    w13 = rng.standard_normal((2 * Is, Hd)) * 0.05
    w2 = rng.standard_normal((Hd, Is)) * 0.05
    if zero:
        w13[:] = 0.0
        w2[:] = 0.0
    q13, s13 = F.quantize_blocks(w13, "e4m3")
    q2, s2 = F.quantize_blocks(w2, "e4m3")
    return [np.ascontiguousarray(a, dtype=np.uint8) for a in (q13, s13, q2, s2)]


def _gpu_shared(B, Hd, Is, codes):
    t = [torch.from_numpy(a).cuda() for a in codes]
    return B.SharedExpert(Hd, Is, *t)


@pytest.mark.parametrize("name,T,Hd,E,k,I,Is,dead_frac", [
    ("sh5", 5, 256, 8, 2, 128, 192, 0.0),          # narrow shared tiles (16 rows)
    ("sh37", 37, 512, 16, 4, 192, 256, 0.25),      # 64-row shared tiles, dead rows
    ("sh300", 300, 256, 8, 2, 128, 576, 0.1),      # wide tiles for both, shared K = 576
])
def test_shared_expert_forward_matches_oracle(name, T, Hd, E, k, I, Is, dead_frac):
    from block_scaled_fp8_moe_gb300 import binding as B
    inp = synth.make_inputs_cpu(synth.custom(name, T, Hd, E, k, I, seed=T + Is, dead_frac=dead_frac))
    g = H.GpuLayer(inp)
    codes = _shared_codes(Hd, Is, seed=T)
    sh = _gpu_shared(B, Hd, Is, codes)
    dead = inp.dead.cuda() if dead_frac > 0 else None
    side = torch.cuda.Stream()
    out = g.forward(dead=dead, shared=sh, side_stream=side)
    same = g.forward(dead=dead, shared=sh)
    torch.cuda.synchronize()
    assert torch.equal(out, same)
    shared_ref = M.SharedExpert(M.DenseWeights(codes[0], codes[1]), M.DenseWeights(codes[2], codes[3]), Is)
    ref, _, _ = H.oracle_forward(inp, use_dead=dead_frac > 0, shared=shared_ref)
    H.assert_out_close(H.bf16_to_np(out), ref.out_exact)
    if dead_frac > 0:
        d = inp.dead.bool().cuda()
        assert torch.all(out[d] == 0)


def test_zero_shared_expert_is_no_shared_expert_and_rows_are_batch_invariant():
    from block_scaled_fp8_moe_gb300 import binding as B
    inp = synth.make_inputs_cpu(synth.custom("sh_inv", 90, 256, 8, 2, 128, seed=9))
    g = H.GpuLayer(inp)
    zero = _gpu_shared(B, 256, 128, _shared_codes(256, 128, seed=1, zero=True))
    plain = g.forward()
    z = g.forward(shared=zero, side_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert torch.equal(z, plain)
    sh = _gpu_shared(B, 256, 128, _shared_codes(256, 128, seed=2))
    full = g.forward(shared=sh).clone()
    for lo, hi in ((0, 1), (7, 40), (89, 90)):
        part = g.forward(x=g.x[lo:hi].contiguous(), shared=sh)
        assert torch.equal(part, full[lo:hi]), (lo, hi)


def test_shared_expert_side_stream_captures_into_a_cuda_graph():
    from block_scaled_fp8_moe_gb300 import binding as B
    inp = synth.make_inputs_cpu(synth.custom("sh_graph", 24, 256, 8, 2, 128, seed=12))
    g = H.GpuLayer(inp)
    sh = _gpu_shared(B, 256, 192, _shared_codes(256, 192, seed=5))
    side = torch.cuda.Stream()
    out = torch.empty(24, 256, dtype=torch.bfloat16, device="cuda")
    ref = g.forward(shared=sh, side_stream=side).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.layer.forward(g.x, out=out, shared=sh, side_stream=side)      # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.layer.forward(g.x, out=out, shared=sh, side_stream=side)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
