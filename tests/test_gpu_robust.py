"""Race and failure-path checks on the GPU: bit-identical results over many calls while another
stream keeps the SMs and HBM busy (the pages' co-resident stress test), and the bounded-wait
timeout path (a wait that nothing completes), after which the context keeps working."""
import pytest
import torch

from block_scaled_fp8_moe_gb300 import synth
from tests import moe_harness as Hh

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,calls", [("decode-6", 12000), ("decode-48", 3000)])
def test_repeat_calls_bit_identical_beside_a_busy_stream(name, calls):
    from block_scaled_fp8_moe_gb300 import binding as B
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs_cuda(cfg)
    layer = B.MoeLayer.from_fp32(inp.w_router, inp.bias, inp.w13, inp.w2, cfg.k)
    del inp.w13, inp.w2
    dead = inp.dead if cfg.dead_frac > 0 else None
    ref = layer.forward(inp.x, dead=dead).clone()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    a = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    out = torch.empty_like(ref)
    for i in range(calls):
        if i % 50 == 0:
            with torch.cuda.stream(side):
                for _ in range(4):
                    a = (a @ a).clamp_(-1, 1)
        layer.forward(inp.x, dead=dead, out=out)
        bad += (out != ref).any().to(torch.int64)
    torch.cuda.synchronize()
    B.moe_check_device_status(layer.workspace(cfg.T))
    assert int(bad.item()) == 0


def test_bounded_wait_expires_reports_and_context_survives():
    from block_scaled_fp8_moe_gb300 import binding as B
    inp = synth.make_inputs_cpu(synth.CONFIGS["tiny"])
    g = Hh.GpuLayer(inp)
    before = g.forward().clone()
    ws = g.layer.workspace(inp.cfg.T)
    B.moe_selftest_timeout(ws, 50_000_000)           # 50 ms wait on a barrier nothing completes
    with pytest.raises(B.MoeError) as ei:
        B.moe_check_device_status(ws)
    assert ei.value.code == B.MOE_ERR_TIMEOUT
    B.moe_check_device_status(ws)                   # the status word was cleared
    after = g.forward()
    assert torch.equal(after, before)
