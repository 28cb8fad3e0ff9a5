"""GPU parity: MX quantisation kernels and the weight packer, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as M

pytestmark = pytest.mark.gpu


def _edge_rows(cols, rng):
    x = rng.standard_normal((12, cols)).astype(np.float32)
    x[0] = 0.0                                    # all-zero blocks -> scale byte 0, codes 0
    x[1] *= 1e-30                                 # tiny values
    x[2] *= 1e30                                  # huge values
    x[3, :32] = 448.0                             # amax exactly at a scale boundary
    x[3, 32:64] = np.float32(448.0 * 1.0078125)   # just above
    x[4] = -0.0                                   # negative zeros
    x[5, ::2] = -x[5, ::2]
    x[6] = rng.choice([-1.0, 1.0], cols) * 2.0 ** rng.integers(-20, 20, cols)
    x[7, :32] = np.float32(1.75) * 2.0 ** -10     # m == 1.75 exactly
    x[8, :32] = 1e-40                             # subnormal amax (fp32)
    return x


@pytest.mark.parametrize("rows,cols", [(1, 32), (7, 256), (129, 4096), (4096, 4096)])
def test_quant_mxfp8_bit_exact(rows, cols):
    from block_scaled_fp8_moe_gb300 import binding as B
    rng = np.random.default_rng(rows * 7 + cols)
    x = rng.standard_normal((rows, cols)).astype(np.float32) * 10.0 ** rng.uniform(-3, 3, (rows, 1))
    if rows >= 12:
        x[:12] = _edge_rows(cols, rng)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    xb = xt.float().numpy()                       # the bf16 values both sides see
    q, s = B.moe_quant_mxfp8(xt.cuda())
    rq, rs = M.quant_mxfp8(xb)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("rows,cols", [(3, 64), (12, 256), (256, 2048)])
def test_quant_mxfp4_bit_exact(rows, cols):
    from block_scaled_fp8_moe_gb300 import binding as B
    rng = np.random.default_rng(rows + cols)
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    if rows >= 12:
        w[:12] = _edge_rows(cols, rng)
    # every E2M1 rounding midpoint at scale 0
    w[0, :14] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0])
    w[0, 14:32] = 6.0
    q, s = B.moe_quant_mxfp4(torch.from_numpy(w).cuda())
    rq, rs = M.quant_mxfp4(w)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("H,I,E", [(256, 128, 3), (512, 576, 2)])
def test_pack_layout(H, I, E):
    """Unpack the packed tiles on the host and compare with the canonical layout."""
    from block_scaled_fp8_moe_gb300 import binding as B
    rng = np.random.default_rng(H + I)
    shp = B.shape(1, H, E, 1, I)
    q13 = rng.integers(0, 256, (E, 2 * I, H // 2), dtype=np.uint8)
    s13 = rng.integers(100, 140, (E, 2 * I, H // 32), dtype=np.uint8)
    q2 = rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8)
    s2 = rng.integers(100, 140, (E, H, I // 32), dtype=np.uint8)
    p13, ps13 = B.moe_pack_w13(shp, torch.from_numpy(q13).cuda(), torch.from_numpy(s13).cuda())
    p2, ps2 = B.moe_pack_w2(shp, torch.from_numpy(q2).cuda(), torch.from_numpy(s2).cuda())
    p13, ps13, p2, ps2 = (t.cpu().numpy() for t in (p13, ps13, p2, ps2))
    for (codes, scales, packed, pscales, gate_up, K) in ((q13, s13, p13, ps13, True, H), (q2, s2, p2, ps2, False, I)):
        MT = I // 64 if gate_up else H // 128
        KC = -(-K // 128)
        tiles = packed.reshape(E, MT, KC, 128, 64)
        stiles = pscales.reshape(E, MT, KC, 512)
        for e in range(E):
            for m in range(MT):
                rows = ([64 * m + r for r in range(64)] + [I + 64 * m + r for r in range(64)]) if gate_up \
                    else [128 * m + r for r in range(128)]
                for kc in range(KC):
                    nb = min(64, K // 2 - kc * 64)
                    want = codes[e, rows, kc * 64: kc * 64 + nb]
                    assert np.array_equal(tiles[e, m, kc, :, :nb], want)
                    assert not tiles[e, m, kc, :, nb:].any()
                    for r in range(128):
                        for b in range(4):
                            blk = kc * 4 + b
                            got = stiles[e, m, kc, (r % 32) * 16 + (r // 32) * 4 + b]
                            assert got == (scales[e, rows[r], blk] if blk < K // 32 else 127)
