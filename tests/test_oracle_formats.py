"""Pins for oracle.formats: E4M3 codes, the round-up exponent rule, bf16 rounding.

Each expected value below comes from the format definition (worked by hand),
from exhaustive enumeration, from brute-force search, from a library cast
(torch.float8_e4m3fn / torch.bfloat16, in-range only), or from facts the
FLAMIA paper prints (tests/golden/paper_facts.json).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "paper_facts.json")))


def test_decode_table_shape():
    vals = F.e4m3_decode_table()
    nan = np.isnan(vals)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    finite = vals[~nan]
    assert finite.size == 254
    assert np.nanmax(vals) == GOLDEN["e4m3_max"]["value"] == 448.0
    assert vals[0x7E] == 448.0 and vals[0xFE] == -448.0
    assert vals[0x01] == 2.0 ** -9                      # smallest subnormal
    assert vals[0x08] == 2.0 ** -6                      # smallest normal
    assert vals[0x38] == 1.0 and vals[0x40] == 2.0
    assert vals[0x80] == 0.0 and math.copysign(1.0, vals[0x80]) == -1.0


def test_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = F.e4m3_encode(F.e4m3_value(codes))
    assert np.array_equal(back, codes)


@pytest.mark.parametrize("v,code", [
    (448.0, 0x7E), (460.0, 0x7E), (464.0, 0x7E), (1e4, 0x7E), (-1e4, 0xFE),   # saturate, never NaN
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (1.5 * 2.0 ** -10, 0x01),          # subnormal, tie to even
    (3 * 2.0 ** -10, 0x02),                                                   # tie between 0x01 and 0x02 -> even
    (1.0625, 0x38), (1.1875, 0x3A), (1.0, 0x38), (-2.0, 0xC0),                # normal ties to even
    (-0.0, 0x80), (0.0, 0x00), (-(2.0 ** -11), 0x80),                          # sign kept through zero
    (240.0, 0x77), (0.5, 0x30), (256.0, 0x78), (416.0, 0x7D),
])
def test_encode_hand_cases(v, code):
    assert int(F.e4m3_encode(np.array([v]))[0]) == code


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200_000) * np.exp2(rng.integers(-14, 9, 200_000))).astype(np.float32)
    x = np.clip(x, -448.0, 448.0)
    ours = F.e4m3_encode(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_neighbour_gap_matches_paper():
    vals = F.e4m3_decode_table()
    pos = np.sort(vals[(~np.isnan(vals)) & (vals >= 2.0 ** -6)])
    gaps = np.diff(pos) / pos[:-1] * 100.0
    g = GOLDEN["e4m3_neighbour_gap_percent"]
    # normal neighbours are between 1/15 and 1/8 apart: the paper rounds the lower end to 7 %
    assert round(gaps.min()) == g["min"] and gaps.max() == g["max"]


@pytest.mark.parametrize("amax,E", [
    (448.0, 0), (450.0, 1), (1.0, -8), (1.75, -8), (1.7578125, -7), (2.0, -7), (896.0, 1), (897.0, 2),
    (0.0, -127), (2.0 ** -130, -127), (2.9e38, 119), (3.0e38, 120),
])
def test_roundup_exponent_hand_cases(amax, E):
    assert int(F.roundup_exponent(np.array([amax]))[0]) == E


def test_roundup_exponent_brute_force():
    rng = np.random.default_rng(1)
    a = np.exp2(rng.uniform(-100, 100, 20000)) * rng.uniform(0.5, 1.0, 20000)
    a = np.concatenate([a, 448.0 * np.exp2(np.arange(-60, 60)), np.nextafter(448.0 * np.exp2(np.arange(-60, 60)), np.inf)])
    E = F.roundup_exponent(a)
    for ai, ei in zip(a[::37], E[::37]):
        cand = [e for e in range(-127, 128) if ai <= 448.0 * 2.0 ** e]
        assert ei == min(cand)
    # vectorised statement of the same property
    assert np.all(a <= 448.0 * np.exp2(E.astype(float)))
    assert np.all(a > 448.0 * np.exp2(E.astype(float) - 1))


def test_floor_rule_can_exceed_448():
    a = np.array([1.9 * 2.0 ** 5, 1.0 * 2.0 ** 5])
    E = F.floor_exponent(a)
    scaled = a / np.exp2(E.astype(float))
    assert scaled[0] > 448.0 and scaled[1] == 256.0
    # the encoder clamps it: the element is no longer represented exactly
    assert F.e4m3_value(F.e4m3_encode(scaled))[0] == 448.0


def test_scale_byte_is_ue8m0():
    assert list(F.scale_byte(np.array([-127, 0, 127]))) == [0, 127, 254]


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100_000) * np.exp2(rng.integers(-40, 40, 100_000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(F.bf16_round(x.astype(np.float64)), ref)
