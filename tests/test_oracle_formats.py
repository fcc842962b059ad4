"""Pins of the oracle's number formats against definitions that do not come from the oracle.

* E2M1 / E4M3 decode: the OCP format definitions (golden fixtures) and torch's independent
  float8_e4m3fn implementation (all 256 codes).
* E4M3 encode: torch's float32 -> float8_e4m3fn conversion (round to nearest even) on a dense
  sweep including every exact midpoint below 448.
* E2M1 encode: hand-worked midpoint table.
* bf16 rounding: torch's float32 -> bfloat16 conversion.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def test_e2m1_value_set_is_ocp_fp4():
    mags = [oracle.e2m1_value(c) for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(8):
        assert oracle.e2m1_value(c | 8) == -mags[c]
    assert math.copysign(1.0, oracle.e2m1_value(8)) == -1.0


def test_e4m3_fixed_points():
    for code, val in _rows("e4m3_points.txt"):
        got = oracle.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert nan.sum() == 2  # only S.1111.111


def test_e4m3_encode_matches_torch_sweep():
    # every representable non-negative value, every midpoint between neighbours, and points just
    # either side of each midpoint, plus a log-spaced sweep, all <= 448 (torch's converter maps
    # overflow to NaN, the oracle saturates; overflow is pinned separately below).
    vals = sorted(set(oracle.e4m3_value(c) for c in range(127)))
    pts = list(vals)
    for a, b in zip(vals[:-1], vals[1:]):
        m = np.float32((a + b) / 2)
        pts += [float(m), float(np.nextafter(m, np.float32(0))), float(np.nextafter(m, np.float32(1e9)))]
    pts += list(np.geomspace(1e-6, 448, 20000, dtype=np.float32).astype(float))
    x = torch.tensor(pts, dtype=torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x.numpy()])
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates():
    for v in (448.0, 449.0, 464.0, 465.0, 1e6, 3.0e38):
        assert oracle.e4m3_encode(v) == 0x7E


def test_e2m1_encode_golden():
    for v, code, *_ in _rows("e2m1_encode_cases.txt"):
        assert oracle.e2m1_encode(float(np.float32(float(v)))) == int(code, 16), v


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(1)
    x = torch.cat([torch.randn(20000, generator=g) * 10 ** torch.randint(-30, 30, (20000,), generator=g),
                   torch.tensor([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3.0e38, 1e-40])])
    x = x.to(torch.float32)
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.double_to_bf16(x.numpy().astype(np.float64))
    assert np.array_equal(ref, got)
