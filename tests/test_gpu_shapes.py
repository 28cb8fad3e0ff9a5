"""GPU parity over a seeded sweep of small and awkward shapes: k = 1, k = E, odd expert counts, the
smallest H and I, I not a multiple of 128 (partial last K-chunk of W2), single rows, more experts
than rows. Routing and plan bit-exact, final output within tolerance of the oracle."""
import numpy as np
import pytest

from block_scaled_fp8_moe_gb300 import synth
from tests import moe_harness as H

pytestmark = pytest.mark.gpu

SHAPES = [
    # T,   H,   E,  k,  I
    (1, 128, 4, 1, 64),
    (3, 128, 3, 3, 64),          # k = E
    (9, 256, 5, 2, 320),         # odd E, I = 320 (2.5 K-chunks)
    (20, 384, 7, 7, 64),         # k = E, 20 rows
    (33, 128, 33, 4, 192),       # E > T
    (70, 256, 12, 1, 448),       # k = 1, 64 < avg rows per expert
    (129, 640, 24, 6, 128),
    (260, 128, 2, 2, 64),        # two experts, every row takes both: 260 rows each (wide tiles)
    (3, 8192, 8, 2, 64),         # widest rows of the decode router (fused quantisation), K = 64 chunks
]


@pytest.mark.parametrize("T,Hd,E,k,I", SHAPES, ids=[f"T{s[0]}H{s[1]}E{s[2]}k{s[3]}I{s[4]}" for s in SHAPES])
def test_shape_sweep_matches_oracle(T, Hd, E, k, I):
    inp = synth.make_inputs_cpu(synth.custom(f"sw{T}_{E}", T, Hd, E, k, I, seed=T * 7 + E))
    g = H.GpuLayer(inp)
    r = g.run_steps()
    ref, _, _ = H.oracle_forward(inp)
    ro = ref.routing
    assert np.array_equal(r["plan"].topk_idx.cpu().numpy(), ro.topk_idx)
    assert np.array_equal(r["plan"].topk_w.cpu().numpy(), ro.topk_w)
    S = int(ro.offsets[-1])
    assert np.array_equal(r["plan"].slot_of_row.cpu().numpy()[:S], ro.slot_of_row)
    bad_q, bad_s = H.e4m3_codes_match(r["hq"].cpu().numpy()[:S], r["hs"].cpu().numpy()[:S], ref.w13.hq,
                                      ref.w13.hs, ref.w13.flip_ok)
    assert bad_q == 0 and bad_s == 0
    H.assert_out_close(H.bf16_to_np(r["out"]), ref.out_exact)
    H.assert_out_close(H.bf16_to_np(g.forward()), ref.out_exact)
