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


def _corrected_quotient(x32, s32):
    """The kernels' division-free quotient in fp32: q0 = x * rcp(s), then q0 - (q0 s - x) rcp(s).
    Both fma steps are emulated in float64: q0 s - x is exact there, and the last step is exact
    to far below an fp32 ulp (enough for these checks)."""
    r = np.float32(1.0) / s32
    q0 = (x32 * r).astype(np.float32)
    rem = (q0.astype(np.float64) * np.float64(s32) - x32.astype(np.float64)).astype(np.float32)
    return (q0.astype(np.float64) - rem.astype(np.float64) * np.float64(r)).astype(np.float32)


def _corrected_quotient_f16(x16, s32):
    """The same quotient in packed fp16, as the full-FP4 PV attention forms it for row values:
    rcp = fp16(fp32 1 / s), q0 = x * rcp, then q0 - (q0 s - x) rcp, each step rounded to fp16
    once (a product of two fp16 values is exact in fp32; the fma steps are exact in float64)."""
    s16 = np.float16(s32)
    r16 = np.float16(np.float32(1.0) / s32)
    q0 = (x16.astype(np.float32) * np.float32(r16)).astype(np.float16)
    rem = (q0.astype(np.float64) * float(s16) - x16.astype(np.float64)).astype(np.float16)
    return (q0.astype(np.float64) - rem.astype(np.float64) * float(r16)).astype(np.float16)


def test_requantisation_of_dequantised_rows_is_exact():
    """The FP4 quantiser and the full-FP4 PV attention round x / s to E2M1 by a division-free
    fp32 quotient and the hardware conversion (nearest, ties to even).  For the values the PV
    variant re-quantises -- dequantised cache values, E2M1 magnitude x positive E4M3 scale --
    against every positive E4M3 scale s:
      * x / s equals a decision point exactly or lies more than 2^-7 (relative) from every one,
        far beyond the quotient's error of an ulp (fp32, or fp16 for the PV variant's rows), so
        the decision is the exact quotient's;
      * at an exact decision point the corrected quotient is exactly that point, and the
        rounding of the emulated quotient equals rounding the exact one everywhere;
      * the level times s is exact and normal in fp16 (the MMA operand format).
    Also: -0 keeps its sign through the quotient."""
    e4 = _e4m3_positive()
    vals = np.unique(np.outer(E2M1_LEVELS, e4).ravel())
    x32 = np.concatenate([vals, -vals]).astype(np.float32)
    assert (np.abs(x32).astype(np.float64) == np.concatenate([vals, vals])).all()
    for s in e4:
        s32 = np.float32(s)
        exact = x32.astype(np.float64) / s
        a = np.abs(exact)
        near = np.min(np.abs(a[:, None] / MIDS[None, :] - 1.0), axis=1)
        on = near == 0.0
        assert (near[~on] > 2.0 ** -7).all(), s
        q = _corrected_quotient(x32, s32)
        assert (np.abs(q[on]).astype(np.float64) == a[on]).all(), s
        assert (_rne_code(q.astype(np.float64)) == _rne_code(exact)).all(), s
        # the PV variant's packed fp16 quotient, for a block's own scale (|x| <= amax <= 6.4 s)
        own = np.abs(x32) <= 6.5 * s
        q16 = _corrected_quotient_f16(x32[own].astype(np.float16), s32)
        assert (np.abs(q16[on[own]]).astype(np.float64) == a[own][on[own]]).all(), s
        assert (_rne_code(q16.astype(np.float64)) == _rne_code(exact[own])).all(), s
        lv = E2M1_LEVELS[_rne_code(exact)] * s
        lv16 = lv.astype(np.float16)
        assert (lv16.astype(np.float64) == lv).all() and (lv[lv > 0] >= 2.0 ** -14).all(), s
    q = _corrected_quotient(np.array([-0.0, 0.0], np.float32), np.float32(0.375))
    assert np.signbit(q).tolist() == [True, False]


def test_corrected_quotient_codes_equal_rounded_quotient_codes():
    """The FP4 quantiser's codes come from the division-free quotient (see above) and the
    hardware E2M1 rounding.  For every finite bf16 value x and every positive E4M3 scale s whose
    quotient stays finite in fp32 (a group's own scale keeps |x / s| below 8, or saturates at 448),
    the rounding of the emulated quotient equals the rounding of the exact one."""
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    for s in _e4m3_positive():
        xs = x[np.abs(x.astype(np.float64) / s) < 2.0 ** 120]
        q = _corrected_quotient(xs, np.float32(s))
        got = _rne_code(q.astype(np.float64))
        ref = _rne_code(xs.astype(np.float64) / s)
        assert (got == ref).all(), (s, xs[got != ref][:5])


def _e4m3_rne(y):
    """Nearest E4M3 value to each y >= 0 (codes 0x00..0x7E), ties to the even code, saturating at
    448: a search over the whole code table."""
    vals = np.concatenate([[0.0], _e4m3_positive()])
    codes = np.arange(0x7F)
    out = []
    for v in np.asarray(y, dtype=np.float64):
        if v >= 448.0:
            out.append(448.0)
            continue
        d = np.abs(vals - v)
        idx = np.nonzero(d == d.min())[0]
        if len(idx) > 1:
            idx = [i for i in idx if codes[i] % 2 == 0]
        out.append(vals[idx[0]])
    return np.array(out)


def test_fp16_block_scale_of_row_values_is_exact():
    """The full-FP4 PV attention computes V's block scales E4M3(fp32(amax / 6)) from fp16 block
    maxima: the fp16 quotient q0 = amax * fp16(1/6), corrected once by the remainder, then the
    hardware E4M3 rounding.  For every possible maximum of dequantised row values (E2M1 magnitude
    x E4M3 scale, and 0) the result equals the rounding of the fp32 quotient, also when q0 is
    one fp16 ulp off either way: the correction, not a lucky rounding, decides the ties (some
    maxima put amax / 6 exactly on an E4M3 midpoint in the subnormal range)."""
    amax = np.unique(np.outer(E2M1_LEVELS, _e4m3_positive()).ravel())
    ref = _e4m3_rne((amax.astype(np.float32) / np.float32(6.0)).astype(np.float64))
    a16 = amax.astype(np.float16)
    assert (a16.astype(np.float64) == amax).all()
    r6 = np.float16(np.float32(1.0) / np.float32(6.0))
    q0 = (a16.astype(np.float32) * np.float32(r6)).astype(np.float16)
    pos = amax > 0
    for step in (0, -1, 1):
        q0p = q0 if step == 0 else np.nextafter(q0, np.float16(np.inf * step)).astype(np.float16)
        rem = (q0p.astype(np.float64) * 6.0 - amax).astype(np.float16)
        q = (q0p.astype(np.float64) - rem.astype(np.float64) * float(r6)).astype(np.float16)
        assert (_e4m3_rne(q[pos].astype(np.float64)) == ref[pos]).all(), step
    ties = np.nonzero(np.abs(amax / 6 / 2.0 ** -9 % 1 - 0.5) == 0)[0]
    assert ties.size > 0  # midpoints of the subnormal quantum occur
