"""The FP4 quantiser's kernel picks each E2M1 code by comparing |x| with exact thresholds T * s
instead of dividing (T = the midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 between neighbouring
E2M1 magnitudes).  This checks, for every bf16 value x and every positive finite E4M3 scale s,
that those comparisons take the same decision as rounding the fp32 quotient x / s to nearest,
ties to the even code -- the rule the oracle states.  Pure numpy: no GPU, no oracle."""
import numpy as np

MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _e4m3_positive():
    """All positive finite E4M3 values (codes 0x01..0x7E), from the format's bit fields."""
    out = []
    for c in range(1, 0x7F):
        e, m = c >> 3, c & 7
        out.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(out)


def _rne_code(q):
    """E2M1 magnitude code of |q| by round to nearest, ties to the even code, saturating."""
    a = np.abs(q)
    return ((a > 0.25).astype(np.int32) + (a >= 0.75) + (a > 1.25) + (a >= 1.75) + (a > 2.5)
            + (a >= 3.5) + (a > 5.0))


def _threshold_code(x, s):
    """The kernel's three comparisons against T * s (fp32)."""
    t = [np.float32(m * s) for m in MIDS]
    assert all(float(ti) == m * s for ti, m in zip(t, MIDS))  # T * s is exact in fp32
    t1, t2, t3, t4, t5, t6, t7 = t
    a = np.abs(x)
    ge4 = a >= t4
    ge2 = a >= np.where(ge4, t6, t2)
    gt1 = a > np.where(ge2, np.where(ge4, t7, t3), np.where(ge4, t5, t1))
    return 4 * ge4.astype(np.int32) + 2 * ge2 + gt1


def test_threshold_codes_equal_rounded_quotient_codes():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)  # every bf16 value, exactly, including signed zeros, inf, NaN
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        for s in _e4m3_positive():
            q = x / np.float32(s)  # correctly rounded fp32 division
            ref = _rne_code(q)
            got = _threshold_code(x, s)
            bad = np.nonzero(ref != got)[0]
            assert bad.size == 0, (s, x[bad[:5]])


def test_ties_go_to_the_even_code():
    s = np.float32(1.0)
    x = MIDS.astype(np.float32)
    assert _threshold_code(x, s).tolist() == [0, 2, 2, 4, 4, 6, 6]


E2M1_LEVELS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _fp16_ladder(a16, s16):
    """The full-FP4 PV attention's re-quantisation of a dequantised row value |v| (fp16) under a
    block scale s (fp16): the level grows by 0.5, 0.5, 0.5, 0.5, 1, 1, 2 as |v| passes the
    decision points T * s (fp16 products), ties to the even code, then is multiplied by s."""
    th = [np.float16(m) * s16 for m in MIDS]
    half, one, two = np.float16(0.5), np.float16(1.0), np.float16(2.0)
    lv = (a16 > th[0]).astype(np.float16) * half
    lv = lv + (a16 >= th[1]).astype(np.float16) * half
    lv = lv + (a16 > th[2]).astype(np.float16) * half
    lv = lv + (a16 >= th[3]).astype(np.float16) * half
    lv = lv + (a16 > th[4]).astype(np.float16) * one
    lv = lv + (a16 >= th[5]).astype(np.float16) * one
    lv = lv + (a16 > th[6]).astype(np.float16) * two
    return th, lv * s16


def test_fp16_requantisation_of_dequantised_rows_is_exact():
    """Every dequantised cache value (E2M1 magnitude x positive E4M3 scale) and every decision
    point T * s is exactly representable as a normal fp16 number, so packed fp16 comparisons
    decide the FP4 code of v / s as rounding the exact quotient does, and the level times s is
    exact too.  Checked for every such value against every positive E4M3 scale."""
    e4 = _e4m3_positive()
    vals = np.unique(np.outer(E2M1_LEVELS, e4).ravel())
    a16 = vals.astype(np.float16)
    assert (a16.astype(np.float64) == vals).all()
    assert (vals[vals > 0] >= 2.0 ** -14).all()  # no fp16 subnormals
    for s in e4:
        s16 = np.float16(s)
        assert float(s16) == s
        th, q = _fp16_ladder(a16, s16)
        assert all(float(t) == m * s and float(t) >= 2.0 ** -14 for t, m in zip(th, MIDS))
        ref = E2M1_LEVELS[_rne_code(vals / s)] * s
        assert (q.astype(np.float64) == ref).all(), s
    # a block of zeros has scale 0 and stays zero
    _, q0 = _fp16_ladder(np.zeros(3, np.float16), np.float16(0.0))
    assert (q0 == 0).all()
