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


# ------------------------------------------------------------------------------------------------
# One-step rounding of doubles to bf16.  The oracle's attention result is a double; it is rounded
# to bf16 once.  Going double -> float -> bf16 instead rounds twice, and a double just above or
# below a bf16 midpoint is then pulled onto the midpoint by the first rounding and sent to the
# even neighbour by the second.  The expected bits come from exact rational arithmetic.
# ------------------------------------------------------------------------------------------------
def _bf16_exact(x: float) -> int:
    """Round the double x to bf16 (8 significant bits, ties to even, subnormal quantum 2^-133,
    overflow to inf) with Python fractions; returns the 16-bit pattern."""
    from fractions import Fraction
    import struct
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    f = Fraction(abs(x))
    e = math.floor(math.log2(abs(x)))
    while Fraction(2) ** e > f:
        e -= 1
    while Fraction(2) ** (e + 1) <= f:
        e += 1
    q = Fraction(2) ** (max(e, -126) - 7)
    n = f / q
    lo = n.numerator // n.denominator
    rem = n - lo
    r = lo + (1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1) else 0)
    val = r * q
    if val >= Fraction(2) ** 128:
        bits = 0x7F80
    else:
        bits = struct.unpack("<I", struct.pack("<f", float(val)))[0] >> 16
    return bits | (0x8000 if x < 0 else 0)


def _near_midpoints():
    """Doubles within 2^-40 (relative) of bf16 midpoints, on both sides, over the normal and the
    subnormal range; none of them is an fp32 value."""
    rng = np.random.default_rng(11)
    xs = []
    for e in list(range(-140, 128, 7)) + [-133, -127, -126, 0, 127]:
        for _ in range(6):
            m = int(rng.integers(0, 128)) if e < -126 else int(rng.integers(128, 256))
            mid = (m + 0.5) * 2.0 ** (max(e, -126) - 7 if e >= -126 else -133)
            for s in (1.0, -1.0):
                for d in (2.0 ** -40, -(2.0 ** -40)):
                    xs.append(s * mid * (1.0 + d))
    return np.array(xs, dtype=np.float64)


def _check_double_to_bf16(fn):
    x = _near_midpoints()
    assert not np.any(x.astype(np.float32).astype(np.float64) == x)  # none is an fp32 value
    want = np.array([_bf16_exact(v) for v in x], dtype=np.uint16)
    got = np.asarray(fn(x), dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {x.size} wrong, e.g. {x[bad[:3]]}"


def test_bf16_rounding_of_doubles_is_one_step():
    _check_double_to_bf16(oracle.double_to_bf16)


def test_bf16_rounding_pin_catches_double_rounding():
    def twice(x):  # the plausible mistake: double -> float -> bf16
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    with pytest.raises(AssertionError):
        _check_double_to_bf16(twice)
