"""Oracle pins for the dead-row rule of the "Speculative decoding" list (post 2 of the flash recipe
thread): a draft row whose estimated chance of surviving verification is below 0.2 skips the
expert weight reads, i.e. it is a dead row of the layer."""
import numpy as np

from oracle import moe as M


def test_threshold_is_the_pages_value():
    assert M.SURVIVAL_THRESHOLD == 0.2


def test_below_threshold_is_dead_at_or_above_is_live():
    # "below 0.2": strictly less, compared in fp32 (fp32(0.2) = 0.20000000298...)
    p = np.array([0.0, np.nextafter(np.float32(0.2), np.float32(0)), 0.2,
                  np.nextafter(np.float32(0.2), np.float32(1)), 1.0, 0.05, 0.7], dtype=np.float32)
    assert M.dead_from_survival(p).tolist() == [1, 1, 0, 0, 0, 1, 0]


def test_special_values():
    p = np.array([np.nan, -np.inf, np.inf, -0.0, -1.0], dtype=np.float32)
    # NaN compares false (the row is computed); -inf and negative estimates are dead; -0 < 0.2
    assert M.dead_from_survival(p).tolist() == [0, 1, 0, 1, 1]


def test_mask_is_monotone_in_the_estimate():
    rng = np.random.default_rng(3)
    p = np.sort(rng.random(1000).astype(np.float32))
    d = M.dead_from_survival(p)
    # sorted ascending: a prefix of dead rows, then live rows, split at the first p >= 0.2
    cut = int(np.searchsorted(p, np.float32(0.2), side="left"))
    assert d[:cut].all() and not d[cut:].any()


def test_custom_threshold_and_layer_effect():
    p = np.array([0.1, 0.3, 0.5], dtype=np.float32)
    assert M.dead_from_survival(p, 0.4).tolist() == [1, 1, 0]
    assert M.dead_from_survival(p, 0.0).tolist() == [0, 0, 0]
    # a dead row takes no plan slot: routing with the derived mask
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    wr = (rng.standard_normal((8, 64)) * 0.02).astype(np.float32)
    bias = np.zeros(8, np.float32)
    r = M.route(x, wr, bias, 2, M.dead_from_survival(p).astype(bool))
    assert int(r.offsets[-1]) == 2 * 2                  # rows 1 and 2 live, k = 2 slots each
    assert (r.row_of_slot[:2] == -1).all()
