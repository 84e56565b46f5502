"""Pins for the oracle's number formats (bf16 and FP8 E4M3), checked against
the format definitions, the pages' printed maximum, and torch's casts."""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def test_e4m3_special_values(oracle_lib):
    o = oracle_lib
    dec = o.e4m3_decode(np.arange(256, dtype=np.uint8))
    # Largest normal printed on the pages ("Formats" section; CS336 notes §5.2).
    assert dec[0x7E] == GOLDEN["e4m3_max_normal"]["value"] == 448.0
    assert dec[0xFE] == -448.0
    assert math.isnan(dec[0x7F]) and math.isnan(dec[0xFF])
    assert np.isnan(dec).sum() == 2          # no infinities, one NaN per sign
    assert dec[0x08] == 2.0 ** -6            # smallest normal
    assert dec[0x01] == 2.0 ** -9            # smallest subnormal
    assert dec[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert dec[0x38] == 1.0                  # exponent field 7 = bias
    assert dec[0x00] == 0.0 and not math.copysign(1.0, dec[0x00]) < 0
    assert dec[0x80] == 0.0 and math.copysign(1.0, dec[0x80]) < 0


def test_e4m3_decode_matches_torch(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle_lib.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])


def test_e4m3_roundtrip_every_code(oracle_lib):
    o = oracle_lib
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = o.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(o.e4m3_encode(vals), codes)


def test_e4m3_ties_go_to_even_code(oracle_lib):
    o = oracle_lib
    pos = np.arange(0x00, 0x7E, dtype=np.uint8)
    lo = o.e4m3_decode(pos)
    hi = o.e4m3_decode(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)       # exact: at most 5 significant bits
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)
    got = o.e4m3_encode(mid)
    want = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    # just either side of a midpoint goes to the nearer code
    above = np.nextafter(mid, np.float32(np.inf))
    below = np.nextafter(mid, np.float32(0))
    assert np.array_equal(o.e4m3_encode(above), (pos + 1).astype(np.uint8))
    assert np.array_equal(o.e4m3_encode(below[1:]), pos[1:])


def test_e4m3_saturates_and_keeps_sign(oracle_lib):
    o = oracle_lib
    big = np.array([448.0, 448.5, 463.9, 464.0, 480.0, 1e4, 3e38, np.inf], np.float32)
    assert np.all(o.e4m3_encode(big) == 0x7E)
    assert np.all(o.e4m3_encode(-big) == 0xFE)
    assert o.e4m3_encode(np.array([np.nan], np.float32))[0] in (0x7F, 0xFF)
    tiny = np.array([1e-30, 2.0 ** -11], np.float32)   # round to zero
    assert np.all(o.e4m3_encode(tiny) == 0x00)
    assert np.all(o.e4m3_encode(-tiny) == 0x80)


def test_e4m3_encode_matches_torch_cast_in_range(oracle_lib):
    rng = np.random.default_rng(123)
    v = np.concatenate([
        rng.uniform(-448, 448, 20000),
        rng.standard_normal(20000) * 0.05,
        rng.standard_normal(20000) * 2.0 ** -8,      # subnormal range
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle_lib.e4m3_encode(v), ref)


def test_e4m3_encode_monotone(oracle_lib):
    v = np.sort(np.random.default_rng(5).uniform(-500, 500, 5000).astype(np.float32))
    dec = oracle_lib.e4m3_decode(oracle_lib.e4m3_encode(v))
    assert np.all(np.diff(dec) >= 0)


def test_bf16_round_matches_torch(oracle_lib):
    rng = np.random.default_rng(7)
    f = np.concatenate([
        rng.standard_normal(50000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),   # subnormals
        rng.uniform(-3e38, 3e38, 5000).astype(np.float32),
    ])
    # exact ties: values with exactly one bit below the bf16 mantissa set
    ties = (rng.integers(0, 1 << 16, 5000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    f = np.concatenate([f, ties[np.isfinite(ties)]])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle_lib.bf16_round(f.astype(np.float64)), ref)


def test_bf16_round_hand_cases(oracle_lib):
    o = oracle_lib
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),          # tie between 1 and 1+2^-7 -> even (1)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),      # tie between 1+2^-7 and 1+2^-6 -> even
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),
        (-2.5, 0xC020),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),              # smallest bf16 subnormal
        (3.4e38, 0x7F80),                   # rounds past the largest finite -> inf
    ]
    for v, bits in cases:
        assert int(o.bf16_round(np.array([v]))[0]) == bits, v
