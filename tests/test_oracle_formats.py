"""Pins for the oracle's number formats (E2M1, E4M3, E8M0).

Checked against: the format tables of the OCP microscaling / FP8 definitions
(hand-worked cases in tests/golden), round trips over every code, monotonicity,
the half-spacing error bound, and torch's own float8_e4m3fn conversion (an
independent library routine) away from saturation.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table():
    for code in range(16):
        mag = E2M1_VALUES[code & 7]
        v = oracle.e2m1_decode(code)
        assert abs(v) == mag
        assert math.copysign(1.0, v) == (-1.0 if code & 8 else 1.0)


def test_e2m1_round_trip_all_codes():
    for code in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_decode(code)) == code


def test_e2m1_hand_worked(golden_dir):
    cases = json.load(open(os.path.join(golden_dir, "e2m1_cases.json")))["cases"]
    for x, code in cases:
        assert oracle.e2m1_encode(x) == code, (x, code)


def test_e2m1_monotone_and_error_bound():
    xs = np.linspace(-8.0, 8.0, 20001)
    dec = np.array([oracle.e2m1_decode(oracle.e2m1_encode(float(x))) for x in xs])
    assert np.all(np.diff(dec) >= 0)
    grid = np.array(sorted(set(E2M1_VALUES + [-v for v in E2M1_VALUES])))
    for x, d in zip(xs, dec):
        if abs(x) >= 6:
            assert abs(d) == 6
            continue
        # the decoded value is a nearest grid point
        assert abs(x - d) <= np.min(np.abs(grid - x)) + 1e-15


def test_e4m3_round_trip_and_order():
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    assert len(finite) == 254
    for c in finite:
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c
    pos = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert np.all(np.diff(pos) > 0)
    assert pos[1] == 2.0 ** -9 and pos[8] == 2.0 ** -6 and pos[0x7E] == 448.0


def test_e4m3_hand_worked(golden_dir):
    cases = json.load(open(os.path.join(golden_dir, "e4m3_cases.json")))["cases"]
    for x, code in cases:
        assert oracle.e4m3_encode(x) == code, (x, code)


def test_e4m3_against_torch_float8():
    g = torch.Generator().manual_seed(7)
    mags = torch.exp(torch.empty(4000, dtype=torch.float64).uniform_(-12.0, 6.0, generator=g))
    sgn = torch.where(torch.rand(4000, generator=g) < 0.5, -1.0, 1.0).double()
    x = (mags * sgn).float()
    x = x[x.abs() <= 448.0]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(v)) for v in x.numpy()], dtype=np.uint8)
    # torch keeps the sign of values that round to zero as well
    assert np.array_equal(ours, ref)


def test_e8m0():
    assert oracle.e8m0_decode(127) == 1.0
    assert oracle.e8m0_decode(0) == 2.0 ** -127
    assert oracle.e8m0_decode(254) == 2.0 ** 127
    assert oracle.e8m0_decode(130) == 8.0
