"""The pooled oracle steps used at full batch size equal the plain oracle calls on the whole batch
(routing and plan, MXFP8 codes, MXFP4 expert weights), on the CPU."""
import numpy as np
import pytest

from block_scaled_fp8_moe_gb300 import synth
from oracle import moe as M
from tests import oracle_pool


@pytest.fixture(scope="module")
def pool():
    with oracle_pool.Pool() as p:
        yield p


def test_pooled_routing_plan_and_quant_equal_the_plain_oracle(pool):
    inp = synth.make_inputs_cpu(synth.custom("pool", 300, 256, 16, 4, 64, seed=3, dead_frac=0.2))
    x = inp.x.float().numpy()
    wr = inp.w_router.float().numpy()
    bias = inp.bias.numpy()
    dead = inp.dead.numpy().astype(bool)
    ref = M.route(x, wr, bias, 4, dead)
    got = pool.route_all(x, wr, bias, 4, dead)
    for f in ("topk_idx", "counts", "offsets", "slot_of_row", "row_of_slot"):
        assert np.array_equal(getattr(got, f), getattr(ref, f)), f
    assert np.array_equal(got.topk_w.view(np.int32), ref.topk_w.view(np.int32))
    q, s = pool.quant_all(x)
    rq, rs = M.quant_mxfp8(x)
    assert np.array_equal(q, rq) and np.array_equal(s, rs)


def test_pooled_weights_equal_plain_quantisation(pool):
    rng = np.random.default_rng(1)
    w = rng.standard_normal((6, 64, 96), dtype=np.float32) * np.float32(0.02)
    ew = pool.weights(lambda e: w[e], 6, 64, 96, [1, 4])
    for e in range(6):
        if e in (1, 4):
            q, s = M.quant_mxfp4(w[e])
            assert np.array_equal(ew.codes[e], q) and np.array_equal(ew.scales[e], s)
        else:
            assert not ew.codes[e].any()
