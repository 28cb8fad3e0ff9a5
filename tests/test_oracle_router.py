"""Pins of the oracle's router: self-written exp/sigmoid, fixed-order logits, top-k, plan."""
import numpy as np
import pytest

from oracle import moe as M


def _ulp(x):
    return np.spacing(np.abs(x).astype(np.float32)).astype(np.float64)


def test_exp_within_two_ulp_of_float64_exp():
    t = np.linspace(-80.0, 80.0, 400001).astype(np.float32)
    got = M.exp_f32(t).astype(np.float64)
    ref = np.exp(t.astype(np.float64))
    assert np.max(np.abs(got - ref) / _ulp(ref)) <= 2.0
    assert M.exp_f32(np.float32([0.0]))[0] == 1.0


def test_sigmoid_within_three_ulp_and_special_values():
    z = np.linspace(-60.0, 60.0, 200001).astype(np.float32)
    got = M.sigmoid_f32(z).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-z.astype(np.float64)))
    assert np.max(np.abs(got - ref) / _ulp(ref)) <= 3.0
    assert M.sigmoid_f32(np.float32([0.0]))[0] == 0.5
    assert M.sigmoid_f32(np.float32([200.0]))[0] == 1.0
    tiny = M.sigmoid_f32(np.float32([-200.0]))[0]       # clamped at -80: exp(-80) region
    assert 0.0 < tiny < 1e-34


def test_bf16_products_are_exact_in_fp32():
    # every pair of bf16 significands (8 bits each), at exponents far apart
    m = (np.arange(128) + 128).astype(np.float64) / 128.0          # 1.0 .. 1.9921875
    for ea, eb in ((0, 0), (-40, 30), (-60, -60), (50, 70)):
        a = (m * 2.0 ** ea).astype(np.float32)
        b = (m * 2.0 ** eb).astype(np.float32)
        p32 = (a[:, None] * b[None, :]).astype(np.float64)
        p64 = a.astype(np.float64)[:, None] * b.astype(np.float64)[None, :]
        assert np.array_equal(p32, p64)


def test_logits_chunked_order_hand_case():
    # h = 0 contributes 1.0; h = 1..127 contribute 2^-25 each. Plain sequential fp32 would stay
    # at 1.0 (each 2^-25 is below half an ulp of 1). In the chunk-of-64 order, chunk 0 gives 1.0,
    # chunk 1 (h = 64..127) gives 64 * 2^-25 = 2^-19 exactly, and 1.0 + 2^-19 is exact.
    H = 128
    x = np.ones((1, H), dtype=np.float32)
    w = np.full((1, H), 2.0 ** -25, dtype=np.float32)
    w[0, 0] = 1.0
    got = M.router_logits(x, w)[0, 0]
    assert got == np.float32(1.0 + 2.0 ** -19)


def test_logits_close_to_exact_dot():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 512)).astype(np.float32)
    w = (rng.standard_normal((7, 512)) * 0.02).astype(np.float32)
    # bf16-exact inputs
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)
    w = (w.view(np.uint32) & 0xFFFF0000).view(np.float32)
    got = M.router_logits(x, w).astype(np.float64)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    bound = (512 + 8) * 2.0 ** -24 * (np.abs(x).astype(np.float64) @ np.abs(w).astype(np.float64).T)
    assert np.all(np.abs(got - exact) <= bound)


def _brute_topk(key, k):
    out = []
    for row in key:
        order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
        out.append(order[:k])
    return np.array(out)


def test_topk_ties_go_to_lower_index():
    key = np.array([[0.5, 0.7, 0.7, 0.1, 0.7, 0.2, 0.5, 0.9]], dtype=np.float32)
    assert M.topk_select(key, 4).tolist() == [[7, 1, 2, 4]]
    rng = np.random.default_rng(1)
    key = rng.integers(0, 4, size=(200, 16)).astype(np.float32)     # many exact ties
    got = M.topk_select(key, 5)
    assert np.array_equal(got, _brute_topk(key, 5))
    # defining property: every selected (key, -e) beats every unselected one
    for t in range(key.shape[0]):
        sel = set(got[t].tolist())
        worst = min(((key[t, e], -e) for e in sel))
        assert all((key[t, e], -e) < worst for e in range(16) if e not in sel)


def test_route_planted_ties_from_duplicate_router_rows():
    rng = np.random.default_rng(2)
    H, E = 128, 8
    x = (rng.standard_normal((6, H)).astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    w = (rng.standard_normal((E, H)).astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    w[5] = w[2]                  # experts 2 and 5 always tie
    bias = np.zeros(E, dtype=np.float32)
    r = M.route(x, w, bias, 3)
    for t in range(6):
        idx = r.topk_idx[t].tolist()
        if 5 in idx:
            assert 2 in idx and idx.index(2) < idx.index(5)


def test_weights_normalised_in_rank_order():
    rng = np.random.default_rng(4)
    H, E, k = 256, 16, 4
    x = (rng.standard_normal((9, H)).astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    w = ((rng.standard_normal((E, H)) * 0.05).astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    r = M.route(x, w, bias, k)
    sel = np.take_along_axis(r.score, r.topk_idx, 1).astype(np.float64)
    assert np.allclose(r.topk_w.sum(1), 1.0, rtol=0, atol=4 * 2.0 ** -24)
    assert np.allclose(r.topk_w, sel / sel.sum(1, keepdims=True), rtol=2 ** -22, atol=0)
    # key = score + bias decides the order, keys non-increasing along rank
    keys = np.take_along_axis(r.key, r.topk_idx, 1)
    assert np.all(np.diff(keys, axis=1) <= 0)


def test_plan_is_a_grouped_permutation_and_dead_rows_take_no_slot():
    rng = np.random.default_rng(5)
    T, E, k = 23, 8, 3
    key = rng.standard_normal((T, E)).astype(np.float32)
    idx = M.topk_select(key, k)
    w = np.full((T, k), 1.0 / k, dtype=np.float32)
    dead = np.zeros(T, dtype=bool)
    dead[[0, 7, 22]] = True
    r = M.plan(key, key, key, idx, w, E, dead)
    live = ~dead
    assert r.counts.sum() == live.sum() * k
    assert r.offsets[0] == 0 and np.all(np.diff(r.offsets) == r.counts)
    # every live slot appears exactly once, dead slots never
    slots = sorted(r.slot_of_row.tolist())
    want = sorted(t * k + j for t in range(T) if live[t] for j in range(k))
    assert slots == want
    for t in range(T):
        for j in range(k):
            p = r.row_of_slot[t * k + j]
            if dead[t]:
                assert p == -1
            else:
                assert r.slot_of_row[p] == t * k + j
                e = idx[t, j]
                assert r.offsets[e] <= p < r.offsets[e + 1]
    # inside an expert, rows ascend in token order
    for e in range(E):
        toks = r.slot_of_row[r.offsets[e]:r.offsets[e + 1]] // k
        assert np.all(np.diff(toks) > 0)


@pytest.mark.parametrize("T", [1, 3])
def test_route_small_batches_are_rowwise(T):
    rng = np.random.default_rng(6)
    H, E = 128, 8
    x = (rng.standard_normal((T, H)).astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    w = ((rng.standard_normal((E, H)) * 0.05).astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    full = M.route(x, w, bias, 2)
    for t in range(T):
        one = M.route(x[t:t + 1], w, bias, 2)
        assert np.array_equal(one.topk_idx[0], full.topk_idx[t])
        assert np.array_equal(one.topk_w[0], full.topk_w[t])
