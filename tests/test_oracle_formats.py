"""Pins of the oracle's number formats against closed forms, a library decoder and brute force."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mx_formats.json")))


def test_e4m3_textbook_values():
    g = GOLD["e4m3"]
    for code, val in g["examples"]:
        got = F.E4M3_TABLE[code]
        assert got == val and np.signbit(got) == np.signbit(val), code
    for c in g["nan_codes"]:
        assert np.isnan(F.E4M3_TABLE[c])
    fin = F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)]
    assert fin.max() == g["max_normal"]
    pos = fin[fin > 0]
    assert pos.min() == g["min_subnormal"]


def test_e4m3_table_matches_torch_decoder():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_TABLE
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.all(both_nan | (ref == ours))
    assert np.array_equal(np.isnan(ref), np.isnan(ours))


def test_e2m1_and_e8m0_textbook_values():
    mags = GOLD["e2m1"]["magnitudes"]
    assert list(F.E2M1_TABLE[:8]) == mags
    assert list(-F.E2M1_TABLE[8:]) == mags
    assert all(np.signbit(F.E2M1_TABLE[8:]))
    for b, val in GOLD["e8m0"]["examples"]:
        assert F.UE8M0_TABLE[b] == val
    assert np.isnan(F.UE8M0_TABLE[GOLD["e8m0"]["nan_code"]])


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_encode_decode_identity_every_finite_code(fmt):
    if fmt == "e4m3":
        codes = np.array([c for c in range(256) if np.isfinite(F.E4M3_TABLE[c])], dtype=np.uint8)
        back = F.encode_e4m3(F.decode_e4m3(codes))
    else:
        codes = np.arange(16, dtype=np.uint8)
        back = F.encode_e2m1(F.decode_e2m1(codes))
    assert np.array_equal(back, codes)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_midpoints_round_to_even_code(fmt):
    table = F.E4M3_TABLE[:127] if fmt == "e4m3" else F.E2M1_TABLE[:8]
    enc = F.encode_e4m3 if fmt == "e4m3" else F.encode_e2m1
    mids = (table[:-1] + table[1:]) / 2.0
    lo_code = np.arange(len(table) - 1)
    want = np.where(lo_code % 2 == 0, lo_code, lo_code + 1)
    assert np.array_equal(enc(mids), want.astype(np.uint8))
    # just off the midpoint goes to the nearer neighbour
    eps = (table[1:] - table[:-1]) * 1e-6
    assert np.array_equal(enc(mids - eps), lo_code.astype(np.uint8))
    assert np.array_equal(enc(mids + eps), (lo_code + 1).astype(np.uint8))
    # negatives mirror
    sign = 0x80 if fmt == "e4m3" else 0x8
    assert np.array_equal(enc(-mids), (want | sign).astype(np.uint8))


def test_e4m3_encode_matches_torch_on_random_values():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(200000) * rng.choice([1e-3, 1e-1, 1, 30, 200], 200000))
    v = np.clip(v, -448, 448).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = F.encode_e4m3(v.astype(np.float64))
    assert np.array_equal(ours, ref)


def test_negative_zero_encodings():
    assert F.encode_e4m3(np.array([-0.0]))[0] == 0x80
    assert F.encode_e2m1(np.array([-0.0]))[0] == 0x8
    assert F.encode_e4m3(np.array([-1e-30]))[0] == 0x80


def test_scale_rule_hand_cases():
    se = F.scale_exponent
    assert se(np.array(448.0), 448.0) == 0
    assert se(np.array(449.0), 448.0) == 1
    assert se(np.array(448.0 * 2 ** -5), 448.0) == -5
    for E in (-20, -3, 0, 7):
        assert se(np.array(1.75 * 2.0 ** E), 448.0) == E - 8
        assert se(np.array(np.nextafter(1.75 * 2.0 ** E, np.inf)), 448.0) == E - 7
        assert se(np.array(1.5 * 2.0 ** E), 6.0) == E - 2
        assert se(np.array(np.nextafter(1.5 * 2.0 ** E, np.inf)), 6.0) == E - 1
    assert se(np.array(6.0), 6.0) == 0
    assert se(np.array(0.0), 448.0) == -127
    assert se(np.array(1e-45), 448.0) == -127      # clamped at the bottom of UE8M0
    assert se(np.array(1e39), 6.0) == 127          # clamped at the top


@pytest.mark.parametrize("qmax", [448.0, 6.0])
def test_scale_rule_is_the_smallest_power_that_fits(qmax):
    rng = np.random.default_rng(3)
    amax = np.abs(rng.standard_normal(100000)) * 10.0 ** rng.uniform(-6, 6, 100000)
    s = F.scale_exponent(amax, qmax)
    assert np.all(amax <= qmax * np.ldexp(1.0, s))
    assert np.all(amax > qmax * np.ldexp(1.0, s - 1))


def test_quantize_blocks_never_saturates_and_is_exact_power_scaling():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 256)) * 10.0 ** rng.uniform(-3, 3, (64, 1))
    for fmt, qmax, dec in (("e4m3", 448.0, F.decode_e4m3), ("e2m1", 6.0, F.decode_e2m1)):
        codes, s = F.quantize_blocks(x, fmt)
        back = F.dequant_blocks(dec(codes), s)
        xb = x.reshape(64, 8, 32)
        # |x * 2^-s| <= qmax in every block
        assert np.all(np.abs(xb) * np.ldexp(1.0, -(s.astype(np.int64) - 127))[..., None] <= qmax)
        # relative error bounded by half an ulp of the element format at the block scale
        mant_bits = 3 if fmt == "e4m3" else 1
        err = np.abs(back - x).reshape(64, 8, 32)
        amax = np.abs(xb).max(-1, keepdims=True)
        assert np.all(err <= amax * 2.0 ** -mant_bits)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(11)
    v = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-30, 30, 100000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = F.f64_to_bf16_bits(v.astype(np.float64))
    assert np.array_equal(ours, ref)


def test_e2m1_nibble_order():
    packed = F.pack_e2m1(np.array([[1, 2, 3, 4]], dtype=np.uint8))
    assert packed.tolist() == [[0x21, 0x43]]
    assert F.unpack_e2m1(packed).tolist() == [[1, 2, 3, 4]]
