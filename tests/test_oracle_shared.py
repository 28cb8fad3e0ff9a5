"""Oracle of the shared expert (TP4 serving profile README: a dense MXFP8 SwiGLU expert on a side
stream beside the routed ones), pinned against the routed path: with one routed expert taking
every row (k = 1, weight exactly 1) and a shared expert holding the same values in MXFP8, the
shared output equals the routed one, so the exact sum doubles. Zero shared weights change nothing;
dead rows stay zero."""
import numpy as np

from oracle import formats as F
from oracle import moe as M


def _layer(T=5, Hd=64, I=64, seed=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, Hd)).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)
    wr = (rng.standard_normal((2, Hd)) * 0.02).astype(np.float32)
    wr = (wr.view(np.uint32) & 0xFFFF0000).view(np.float32)
    bias = np.array([100.0, -100.0], np.float32)                 # every row picks expert 0
    w13 = np.zeros((2, 2 * I, Hd // 2), np.uint8), np.zeros((2, 2 * I, Hd // 32), np.uint8)
    w2 = np.zeros((2, Hd, I // 2), np.uint8), np.zeros((2, Hd, I // 32), np.uint8)
    for e in range(2):
        w13[0][e], w13[1][e] = M.quant_mxfp4(rng.standard_normal((2 * I, Hd)) * 0.05)
        w2[0][e], w2[1][e] = M.quant_mxfp4(rng.standard_normal((Hd, I)) * 0.05)
    return x, wr, bias, M.ExpertWeights(*w13), M.ExpertWeights(*w2), I


def _as_mxfp8(ew: M.ExpertWeights, e: int) -> M.DenseWeights:
    # an MXFP4 value has at most two significant bits, so MXFP8 holds it exactly
    vals = ew[e]
    q, s = F.quantize_blocks(vals, "e4m3")
    dw = M.DenseWeights(q, s)
    assert np.array_equal(dw[0], vals)
    return dw


def test_shared_equal_to_the_routed_expert_doubles_the_sum():
    x, wr, bias, w13, w2, I = _layer()
    plain = M.forward(x, wr, bias, 1, w13, w2, I)
    assert np.all(plain.routing.topk_idx == 0) and np.all(plain.routing.topk_w == 1.0)
    sh = M.SharedExpert(_as_mxfp8(w13, 0), _as_mxfp8(w2, 0), I)
    both = M.forward(x, wr, bias, 1, w13, w2, I, shared=sh)
    assert np.array_equal(both.out_exact, 2.0 * plain.out_exact)


def test_zero_shared_weights_change_nothing_and_dead_rows_stay_zero():
    x, wr, bias, w13, w2, I = _layer(T=6, seed=4)
    Hd = x.shape[1]
    zero = M.SharedExpert(M.DenseWeights(np.zeros((2 * I, Hd), np.uint8), np.full((2 * I, Hd // 32), 127, np.uint8)),
                          M.DenseWeights(np.zeros((Hd, I), np.uint8), np.full((Hd, I // 32), 127, np.uint8)), I)
    plain = M.forward(x, wr, bias, 1, w13, w2, I)
    z = M.forward(x, wr, bias, 1, w13, w2, I, shared=zero)
    assert np.array_equal(z.out_exact, plain.out_exact)
    dead = np.zeros(6, bool)
    dead[[1, 4]] = True
    sh = M.SharedExpert(_as_mxfp8(w13, 1), _as_mxfp8(w2, 1), I)
    d = M.forward(x, wr, bias, 1, w13, w2, I, dead=dead, shared=sh)
    assert np.all(d.out[dead] == 0.0) and not np.any(np.signbit(d.out[dead]))
    full = M.forward(x, wr, bias, 1, w13, w2, I, shared=sh)
    assert np.array_equal(d.out[~dead], full.out[~dead])
