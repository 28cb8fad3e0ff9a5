"""Pins of the oracle's whole layer: closed forms, exact brute force, invariances."""
import math
from fractions import Fraction

import numpy as np
import pytest

from block_scaled_fp8_moe_gb300 import synth
from oracle import formats as F
from oracle import moe as M


def _weights(w):
    """fp32 [E, R, K] -> oracle ExpertWeights (canonical MXFP4)."""
    E, R, K = w.shape
    q, s = M.quant_mxfp4(np.asarray(w, dtype=np.float32).reshape(E * R, K))
    return M.ExpertWeights(q.reshape(E, R, K // 2), s.reshape(E, R, K // 32), cache=64)


def _const_weights(E, R, K, code, scale_byte=127):
    q = np.full((E, R, K // 2), (code & 0xF) | ((code & 0xF) << 4), dtype=np.uint8)
    s = np.full((E, R, K // 32), scale_byte, dtype=np.uint8)
    return M.ExpertWeights(q, s, cache=64)


def _bf16(a):
    return (np.asarray(a, dtype=np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)


def test_all_ones_closed_form():
    # x = 1, every weight = 1.0: g = u = H, a = H * sigmoid(H) * H = H^2 (sigmoid(256) rounds to 1),
    # requant of H^2 is exact, y_j = w_j * I * H^2, and the weights sum to one -> out = I * H^2.
    H, I, E, k, T = 256, 128, 8, 2, 3
    x = np.ones((T, H), dtype=np.float32)
    rng = np.random.default_rng(0)
    wr = _bf16(rng.standard_normal((E, H)) * 0.02)
    bias = np.zeros(E, dtype=np.float32)
    w13 = _const_weights(E, 2 * I, H, 0x2)
    w2 = _const_weights(E, H, I, 0x2)
    r = M.forward(x, wr, bias, k, w13, w2, I)
    assert np.all(r.w13.a == float(H * H))
    assert np.all(r.out == float(I * H * H))


def test_gate_and_up_are_not_swapped_closed_form():
    # gate rows = -1, up rows = +1, x = 1/64: g = -H/64, u = H/64, a = g * sigmoid(g) * u.
    H, I, E, k = 256, 64, 4, 1
    x = np.full((2, H), 1.0 / 64, dtype=np.float32)
    wr = _bf16(np.random.default_rng(1).standard_normal((E, H)) * 0.02)
    q = np.zeros((E, 2 * I, H // 2), dtype=np.uint8)
    q[:, :I] = 0xAA           # -1.0 in both nibbles
    q[:, I:] = 0x22           # +1.0
    s = np.full((E, 2 * I, H // 32), 127, dtype=np.uint8)
    w13 = M.ExpertWeights(q, s)
    w2 = _const_weights(E, H, I, 0x2)
    r = M.forward(x, wr, np.zeros(E, np.float32), k, w13, w2, I)
    g, u = -H / 64.0, H / 64.0
    want = g / (1.0 + math.exp(-g)) * u
    assert np.allclose(r.w13.a, want, rtol=1e-15, atol=0)


def test_dropped_or_misplaced_weight_block_changes_the_result():
    # one weight 32-block with a different scale must move exactly the rows it belongs to
    H, I, E, k = 256, 64, 2, 1
    x = np.ones((1, H), dtype=np.float32)
    wr = np.zeros((E, H), dtype=np.float32)      # all keys equal -> expert 0 (lowest index)
    w13 = _const_weights(E, 2 * I, H, 0x2)
    w13.scales[0, 3, 5] = 128                    # gate row 3, K block 5 doubled
    w2 = _const_weights(E, H, I, 0x2)
    r = M.forward(x, wr, np.zeros(E, np.float32), k, w13, w2, I)
    g = np.full(I, float(H))
    g[3] += 32.0
    u = float(H)
    want = g / (1.0 + np.exp(-g)) * u
    assert np.array_equal(r.w13.a[0], want)


def _exact_dot(wrow_codes, wrow_scales, xhat_frac, nib):
    """Exact rational dot of one MXFP4 row with exact activations."""
    acc = Fraction(0)
    K = len(xhat_frac)
    for kk in range(K):
        c = nib[kk]
        if c & 7 == 0:
            continue
        v = Fraction(F.E2M1_TABLE[c]).limit_denominator(4) * (Fraction(2) ** (int(wrow_scales[kk // 32]) - 127))
        acc += v * xhat_frac[kk]
    return acc


def test_tiny_config_against_exact_rational_brute_force():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs_cpu(cfg)
    x = inp.x.float().numpy()
    wr = inp.w_router.float().numpy()
    bias = inp.bias.numpy()
    w13 = _weights(inp.w13.numpy())
    w2 = _weights(inp.w2.numpy())
    r = M.forward(x, wr, bias, cfg.k, w13, w2, cfg.I)
    xq, xs = r.xq, r.xs
    # Brute force: loop tokens and their top-k directly (no plan), exact rationals for the sums.
    for t in range(cfg.T):
        xhat = [Fraction(float(v)) for v in M.decode_mxfp8(xq[t], xs[t])]
        acc = np.zeros(cfg.H)
        for j in range(cfg.k):
            e = int(r.routing.topk_idx[t, j])
            p = r.routing.row_of_slot[t * cfg.k + j]
            n = int(np.nonzero(r.w13.rows == p)[0][0])
            nib13 = F.unpack_e2m1(w13.codes[e])
            a = np.zeros(cfg.I)
            for i in range(cfg.I):
                g = float(_exact_dot(w13.codes[e][i], w13.scales[e][i], xhat, nib13[i]))
                u = float(_exact_dot(w13.codes[e][cfg.I + i], w13.scales[e][cfg.I + i], xhat, nib13[cfg.I + i]))
                a[i] = g / (1.0 + math.exp(-g)) * u
            assert np.allclose(r.w13.a[n], a, rtol=1e-12, atol=1e-300)
            hhat = [Fraction(float(v)) for v in M.decode_mxfp8(r.w13.hq[n], r.w13.hs[n])]
            nib2 = F.unpack_e2m1(w2.codes[e])
            y = np.array([float(_exact_dot(w2.codes[e][o], w2.scales[e][o], hhat, nib2[o]))
                          for o in range(cfg.H)])
            acc = acc + np.float64(r.routing.topk_w[t, j]) * y
        want = F.round_to_bf16(acc)
        got = r.out[t]
        # float64 vs exact sums can only move a bf16 rounding by one step
        step = np.ldexp(1.0, np.frexp(np.abs(want))[1] - 8)
        assert np.all(np.abs(got - want) <= step)


def _tiny_layer(T=6, seed=3, H=256, I=128, E=8, k=2):
    cfg = synth.custom("t", T, H, E, k, I, seed)
    inp = synth.make_inputs_cpu(cfg)
    return (cfg, inp.x.float().numpy(), inp.w_router.float().numpy(), inp.bias.numpy(),
            _weights(inp.w13.numpy()), _weights(inp.w2.numpy()))


def test_oracle_rows_do_not_depend_on_the_batch():
    cfg, x, wr, bias, w13, w2 = _tiny_layer()
    full = M.forward(x, wr, bias, cfg.k, w13, w2, cfg.I)
    for t in range(cfg.T):
        one = M.forward(x[t:t + 1], wr, bias, cfg.k, w13, w2, cfg.I)
        assert np.array_equal(one.out[0], full.out[t])
    perm = np.random.default_rng(0).permutation(cfg.T)
    shuf = M.forward(x[perm], wr, bias, cfg.k, w13, w2, cfg.I)
    assert np.array_equal(shuf.out, full.out[perm])


def test_dead_rows_are_zero_and_leave_live_rows_unchanged():
    cfg, x, wr, bias, w13, w2 = _tiny_layer()
    dead = np.zeros(cfg.T, dtype=bool)
    dead[[1, 4]] = True
    full = M.forward(x, wr, bias, cfg.k, w13, w2, cfg.I)
    d = M.forward(x, wr, bias, cfg.k, w13, w2, cfg.I, dead=dead)
    assert np.all(d.out[dead] == 0.0) and not np.any(np.signbit(d.out[dead]))
    assert np.array_equal(d.out[~dead], full.out[~dead])
    assert int(d.routing.offsets[-1]) == (cfg.T - 2) * cfg.k
    assert np.array_equal(d.routing.topk_idx, full.routing.topk_idx)


def test_sampled_tokens_match_full_forward():
    cfg, x, wr, bias, w13, w2 = _tiny_layer(T=9)
    full = M.forward(x, wr, bias, cfg.k, w13, w2, cfg.I)
    part = M.forward(x, wr, bias, cfg.k, w13, w2, cfg.I, tokens=np.array([2, 7]))
    assert np.array_equal(part.out, full.out[[2, 7]])


def test_flip_eligibility_marks_boundaries():
    a = np.zeros((1, 32))
    a[0, 0] = 448.0                  # amax exactly at the scale boundary
    a[0, 1] = 1.0625                 # midpoint between E4M3 1.0 and 1.125 at scale 0
    a[0, 2] = 1.0
    ok = M.requant_flip_eligible(a, 1e-5)
    assert ok[0, 0] and ok[0, 1]     # the whole block may rescale; the midpoint may round either way
    b = np.zeros((1, 32))
    b[0, 0] = 392.0
    b[0, 1] = 1.0625
    b[0, 2] = 1.0
    ok = M.requant_flip_eligible(b, 1e-5)
    assert ok[0, 1] and not ok[0, 2] and not ok[0, 0]
