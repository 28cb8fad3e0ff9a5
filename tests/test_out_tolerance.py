"""The final-output check of the parity tests (CPU): the bf16 output must be the RNE rounding of a
value within 2e-2 x rms of the oracle's exact sum, so a flip of the last bf16 bit at a rounding
boundary passes while a real error of the same size elsewhere does not."""
import numpy as np
import pytest

from tests import moe_harness as H
from oracle import formats as F
from oracle import moe as M


def test_combine_rounds_combine_exact():
    rng = np.random.default_rng(3)
    y = {s: rng.standard_normal(64) for s in range(12) if s != 5}     # slot 5 absent
    ex = M.combine_exact(y, 4, 3, 64, np.arange(4))
    out = M.combine(y, 4, 3, 64, np.arange(4))
    assert np.array_equal(out, F.round_to_bf16(ex) + 0.0)
    assert np.array_equal(ex[1], (y[3] + y[4]) + 0.0)                 # token 1: slots 3, 4 (5 dead)


def test_boundary_flip_passes_real_error_fails():
    q = 2.0 ** -11                             # bf16 quantum on [2^-4, 2^-3)
    rng = np.random.default_rng(4)
    ex = rng.standard_normal(4096) * 0.005     # rms ~0.005: tolerance 1e-4 ~ 0.2 quantum
    tol = 2e-2 * np.sqrt(np.mean(ex ** 2))
    assert tol < q / 2
    ex[0] = 205.5 * q + 1e-9                   # just above the midpoint of 205 q and 206 q
    got = F.round_to_bf16(ex)
    assert got[0] == 206 * q
    H.assert_out_close(got, ex)                # exact rounding passes
    flip = got.copy()
    flip[0] = 205 * q                          # the other side of the boundary: a flip
    H.assert_out_close(flip, ex)
    ex2 = ex.copy()
    ex2[0] = 205.25 * q                        # rounds to 205 q, a quarter quantum from the midpoint
    far = F.round_to_bf16(ex2)
    H.assert_out_close(far, ex2)
    far[0] = 204 * q                           # one quantum off away from any boundary: an error
    with pytest.raises(AssertionError):
        H.assert_out_close(far, ex2)
