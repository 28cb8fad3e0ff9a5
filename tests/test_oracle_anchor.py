"""Anchored verify rows (TP4 serving profile README, settings table row "Verify length"): a row
whose anchor is a reuses that row's experts -- so the set of experts a batch touches does not grow
-- and weights them with its own sigmoid scores. Pinned against the plain top-k router and a
brute-force recomputation of the weights."""
import numpy as np
import pytest

from oracle import moe as M


def _inputs(t=12, h=128, e=16, seed=7):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((t, h)).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)          # bf16 values
    wr = (rng.standard_normal((e, h)) * 0.05).astype(np.float32)
    wr = (wr.view(np.uint32) & 0xFFFF0000).view(np.float32)
    bias = (rng.standard_normal(e) * 0.1).astype(np.float32)
    return x, wr, bias


def test_no_anchor_is_plain_routing():
    x, wr, bias = _inputs()
    a = M.route(x, wr, bias, 4)
    b = M.route(x, wr, bias, 4, anchor=np.full(12, -1))
    assert np.array_equal(a.topk_idx, b.topk_idx) and np.array_equal(a.topk_w, b.topk_w)
    assert np.array_equal(a.slot_of_row, b.slot_of_row)


def test_anchored_rows_take_the_anchor_experts_with_their_own_scores():
    x, wr, bias = _inputs()
    x[4] = x[0]                                                  # row 4 duplicates its anchor
    k = 4
    anchor = np.full(12, -1)
    anchor[[3, 4, 9]] = [0, 0, 7]
    plain = M.route(x, wr, bias, k)
    r = M.route(x, wr, bias, k, anchor=anchor)
    for t in range(12):
        src = anchor[t] if anchor[t] >= 0 else t
        assert np.array_equal(r.topk_idx[t], plain.topk_idx[src])
        if anchor[t] < 0:
            assert np.array_equal(r.topk_w[t], plain.topk_w[t])
    # a duplicate of its anchor gets exactly the anchor's weights
    assert np.array_equal(r.topk_w[4], plain.topk_w[0])
    # weights are the row's own scores of the anchor's experts, normalised: they sum to 1 and
    # keep the ratios of those scores
    for t in (3, 9):
        s = plain.score[t, r.topk_idx[t]].astype(np.float64)
        w = r.topk_w[t].astype(np.float64)
        assert abs(w.sum() - 1.0) < 1e-6
        assert np.allclose(w / w[0], s / s[0], rtol=1e-6)
    # rows 3, 4 and 9 do not reach any expert outside what their anchors reach
    touched_plain_anchors = set(plain.topk_idx[[0, 7]].ravel().tolist())
    assert set(r.topk_idx[[3, 4, 9]].ravel().tolist()) <= touched_plain_anchors


def test_anchors_never_grow_the_touched_expert_set():
    x, wr, bias = _inputs(t=40, e=32, seed=11)
    k = 3
    anchor = np.full(40, -1)
    anchor[20:] = np.arange(20) % 5                              # rows 20.. reuse rows 0..4
    r = M.route(x, wr, bias, k, anchor=anchor)
    alone = M.route(x[:20], wr, bias, k)
    assert set(np.nonzero(r.counts)[0].tolist()) == set(np.nonzero(alone.counts)[0].tolist())


def test_anchor_validation():
    x, wr, bias = _inputs()
    with pytest.raises(ValueError):
        M.route(x, wr, bias, 4, anchor=np.full(11, -1))           # wrong length
    bad = np.full(12, -1)
    bad[2] = 12
    with pytest.raises(ValueError):
        M.route(x, wr, bias, 4, anchor=bad)                       # out of range
    chain = np.full(12, -1)
    chain[2], chain[3] = 1, 2
    with pytest.raises(ValueError):
        M.route(x, wr, bias, 4, anchor=chain)                     # anchor row itself anchored
