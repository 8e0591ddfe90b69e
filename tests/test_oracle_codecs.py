"""Pins of the oracle's codecs against library routines and hand-derived values.

The oracle's encoders are written from the format definitions (enumeration of
representable values); here they are checked against PyTorch's own fp8/e8m0
conversions (a library routine, independent of the oracle) and against values
derived by hand from the OCP MX formats (E4M3FN, E2M1, UE8M0).
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.e4m3_values()
    nan = np.isnan(ref)
    assert (nan == np.isnan(ours)).all()
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert (ref[~nan] == ours[~nan]).all()
    # hand-derived anchors: max normal, min normal, min subnormal
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0xFE) == -448.0


def _all_bf16_below(limit):
    u = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    f = u.view(np.float32)
    keep = np.isfinite(f) & (np.abs(f) < limit)
    return f[keep]


def test_e4m3_encode_exhaustive_bf16_vs_torch():
    # Every finite bf16 value below 448 in magnitude (RNE, ties to even, -0 kept).
    x = _all_bf16_below(448.0)
    ours = oracle.e4m3_encode_array(x.astype(np.float64))
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (ours == ref).all(), np.flatnonzero(ours != ref)[:10]


def test_e4m3_encode_ties_and_saturation():
    # 400 lies exactly between 384 (m=4) and 416 (m=5): ties go to the even code.
    assert oracle.e4m3_encode(400.0) == 0x7C
    # half the smallest subnormal rounds to zero (even), just above it rounds up
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(2.0 ** -10 * 1.0001) == 0x01
    # largest subnormal / smallest normal midpoint goes to the even (normal) code
    assert oracle.e4m3_encode((7 / 8 * 2 ** -6 + 2 ** -6) / 2) == 0x08
    assert oracle.e4m3_encode(-12.0) == 0xD4
    assert oracle.e4m3_encode(1e6) == 0x7E


def test_e4m3_roundup_minimal():
    rng = random.Random(7)
    vals = oracle.e4m3_values()
    for _ in range(3000):
        r = math.ldexp(rng.random() + 0.5, rng.randint(-12, 8))
        if r >= 448:
            continue
        c = oracle.e4m3_roundup(r)
        assert vals[c] >= r
        assert c == 1 or vals[c - 1] < r
    assert oracle.e4m3_roundup(448.0) == 0x7E
    assert oracle.e4m3_roundup(1.0) == 0x38
    assert oracle.e4m3_roundup(1.0000001) == 0x39
    assert oracle.e4m3_roundup(0.0) == 0


E2M1_HAND = {  # value -> code, from the E2M1 definition (bias 1, one mantissa bit), RNE
    0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7,
    0.25: 0,   # tie 0 / 0.5 -> even code 0
    0.75: 2,   # tie 0.5 (code 1) / 1.0 (code 2) -> 2
    1.25: 2,   # tie 1.0 / 1.5 -> 2
    1.75: 4,   # tie 1.5 / 2.0 -> 4
    2.5: 4,    # tie 2 / 3 -> 4
    3.5: 6,    # tie 3 / 4 -> 6
    5.0: 6,    # tie 4 / 6 -> 6
    5.1: 7, 4.9: 6, 0.26: 1, 10.0: 7,
    -1.5: 11, -6.0: 15, -0.1: 8,
}


@pytest.mark.parametrize("x,code", sorted(E2M1_HAND.items()))
def test_e2m1_encode_hand_values(x, code):
    assert oracle.e2m1_encode(x) == code


def test_e2m1_encode_is_nearest():
    vals = np.array([oracle.e2m1_decode(c) for c in range(8)])
    xs = np.linspace(0, 6, 20001)
    codes = oracle.e2m1_encode_array(xs)
    err = np.abs(vals[codes] - xs)
    best = np.min(np.abs(vals[None, :] - xs[:, None]), axis=1)
    assert np.allclose(err, best, rtol=0, atol=0)


def test_ue8m0_decode_matches_torch():
    b = torch.arange(255, dtype=torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    ours = np.array([oracle.ue8m0_decode(i) for i in range(255)])
    assert (ref == ours).all()
    assert math.isnan(oracle.ue8m0_decode(255))


@pytest.mark.parametrize("amax,e", [(448.0, 0), (449.0, 1), (1.0, -8), (0.875, -9), (1.75, -8),
                                    (1.7500001, -7), (100.0, -2), (0.002, -17), (0.0, 0),
                                    (2.0 ** -140, -148)])
def test_noclamp_exponent_hand_values(amax, e):
    assert oracle.noclamp_exponent(amax) == e


def test_noclamp_exponent_is_smallest_nonclamping():
    # definition: smallest integer e with amax <= 448 * 2^e (checked in exact rationals)
    rng = np.random.default_rng(3)
    xs = np.ldexp(rng.random(20000) + 0.5, rng.integers(-60, 60, 20000))
    es = oracle.noclamp_exponent_array(xs)
    for x, e in zip(xs[:4000], es[:4000]):
        fx = Fraction(float(x))
        assert fx <= 448 * Fraction(2) ** int(e)
        assert fx > 448 * Fraction(2) ** (int(e) - 1)


def test_scale_exponent_clamps_to_ue8m0_range():
    assert oracle.scale_exponent(1e-45) == -127
    assert oracle.scale_exponent(3.0e38) == 120


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(50000) * np.exp(rng.uniform(-20, 20, 50000))
    ref = torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    ours = np.array([oracle.round_bf16(v) for v in x])
    assert (ref == ours).all()
