"""The kernels' zero-order-hold factor E = (exp(x) - 1) / a, x = dt a (dpshk.com/news/3333417 section 2.2),
restated on the CPU in fp32 arithmetic step by step as the device code forms it, and checked against
libm's expm1 in fp64.  The coefficients and thresholds are read from the device header, so a change
there is checked here.

Formed as (Abar - 1) / a, E loses accuracy as |x| -> 0; the device code switches to the Taylor series of
expm1(x) / x below |x| = 2^-4.  The checks: the coefficients are (ln 2)^k / (k+1)!; E (and dE/da for the
backward pass) is within a few 1e-7 relative over the series range, within 1e-5 above it when Abar
carries the 2-ulp error of the hardware exp2; and the plain quotient, planted in place of the series,
fails the same check (so the check can tell the two apart).  dE/da switches to its series below
|x| = 1/4, where dt Abar - E would cancel."""
import math
import os
import re

import numpy as np
import pytest

HEADER = os.path.join(os.path.dirname(__file__), "..", "selective_state_space_156_b300", "csrc", "ssm_device.cuh")
f32 = np.float32


def _const(name):
    text = open(HEADER).read()
    m = re.search(r"constexpr float %s = ([^;/]+);" % name, text)
    assert m, name
    expr = m.group(1).strip().replace("kLog2e", "1.4426950408889634f")
    # "0.0625f * 1.44...f" or a literal
    val = 1.0
    for part in expr.split("*"):
        val *= float(part.strip().rstrip("f"))
    return f32(val)


PHI1, PHI2, PHI3 = _const("kPhiY1"), _const("kPhiY2"), _const("kPhiY3")
SERIES_Y = _const("kZohSeriesY")
SERIES_X = _const("kZohSeriesX")
SERIES_DA_X = _const("kZohDaSeriesX")
LOG2E = f32(1.4426950408889634)


def fma32(a, b, c):
    # the product of two fp32 values is exact in fp64; one rounding to fp32 at the end (as fmaf)
    return f32(float(a) * float(b) + float(c))


def ex2_approx(y, ulps):
    """2^y rounded to fp32, then moved by `ulps` units in the last place (the hardware's approximation)."""
    r = f32(2.0 ** float(y))
    return np.nextafter(r, f32(np.inf) if ulps > 0 else f32(-np.inf)) if ulps else r


def device_E(dt, a, ulps=0, series=True):
    """E as the device forms it (zoh_factor): y = dt (a log2 e), ab = 2^y, the series below the threshold."""
    dt, a = f32(dt), f32(a)
    y = f32(dt * f32(a * LOG2E))
    ab = ex2_approx(y, ulps)
    inva = f32(1.0) / a if a != 0 else f32(0.0)
    big = f32(f32(ab - f32(1.0)) * inva)
    p = fma32(y, PHI3, PHI2)
    p = fma32(p, y, PHI1)
    p = fma32(p, y, f32(1.0))
    small = f32(dt * p)
    return (small if (series and abs(y) < SERIES_Y) else big), ab


def device_dEda(dt, a, ulps=0):
    """dE/da as the backward pass forms it (zoh_factor_da)."""
    E, ab = device_E(dt, a, ulps)
    dt, a = f32(dt), f32(a)
    x = f32(dt * a)
    inva = f32(1.0) / a if a != 0 else f32(0.0)
    big = f32(fma32(dt, ab, -E) * inva)
    p = fma32(x, f32(1.0 / 840.0), f32(1.0 / 144.0))
    p = fma32(p, x, f32(1.0 / 30.0))
    p = fma32(p, x, f32(0.125))
    p = fma32(p, x, f32(1.0 / 3.0))
    p = fma32(p, x, f32(0.5))
    small = f32(f32(dt * dt) * p)
    return small if abs(x) < SERIES_DA_X else big


def exact_E(dt, a):
    dt, a = float(f32(dt)), float(f32(a))
    return dt if a == 0 else math.expm1(dt * a) / a


def exact_dEda(dt, a):
    dt, a = float(f32(dt)), float(f32(a))
    x = dt * a
    if abs(x) < 1e-3:  # the series of dt^2 phi'(x) to x^5 in fp64 (truncation < 1e-19 relative)
        return dt * dt * (0.5 + x / 3 + x * x / 8 + x ** 3 / 30 + x ** 4 / 144 + x ** 5 / 840)
    return (dt * math.exp(x) - math.expm1(x) / a) / a


def test_coefficients_are_the_taylor_series_of_expm1_over_x():
    ln2 = math.log(2.0)
    for k, c in ((1, PHI1), (2, PHI2), (3, PHI3)):
        assert abs(float(c) - ln2 ** k / math.factorial(k + 1)) <= 1e-7 * float(c)
    text = open(HEADER).read()
    body = text[text.index("float zoh_factor_da("):]
    body = body[:body.index("}")]
    # phi'(x) coefficients k / (k+1)! for k = 1..6, highest first as Horner takes them
    want = [k / math.factorial(k + 1) for k in range(6, 0, -1)]
    nums = re.findall(r"1\.0f / ([0-9.]+)f|, (0\.125)f|, (0\.5)f", body)
    vals = [1.0 / float(a) if a else float(b or c) for a, b, c in nums]
    assert np.allclose(vals, want, rtol=1e-7), (vals, want)
    assert abs(float(SERIES_Y) - float(SERIES_X) / math.log(2.0)) < 1e-6
    assert float(SERIES_X) == 2.0 ** -4


def _grid():
    """(dt, a) pairs covering x = dt a over [-2^-4, 0] densely, across the threshold, and far beyond."""
    xs = -np.concatenate([np.geomspace(1e-9, 2.0 ** -4, 400), np.geomspace(2.0 ** -4, 40.0, 200)])
    out = []
    for i, x in enumerate(xs):
        dt = (1e-4, 1e-3, 1e-2, 1e-1)[i % 4]
        out.append((dt, x / dt))
    return out


@pytest.mark.parametrize("ulps", [0, 2, -2])
def test_E_matches_libm(ulps):
    worst_series = worst_quot = 0.0
    for dt, a in _grid():
        got, _ = device_E(dt, a, ulps)
        want = exact_E(dt, a)
        rel = abs(float(got) - want) / abs(want)
        x = abs(float(f32(dt)) * float(f32(a)))
        if x < 2.0 ** -4 * 0.999:
            worst_series = max(worst_series, rel)
        elif x > 2.0 ** -4 * 1.001:
            worst_quot = max(worst_quot, rel)
    assert worst_series < 3e-7, worst_series
    assert worst_quot < 1e-5, worst_quot


def test_E_at_zero_A_is_dt():
    for dt in (1e-4, 1e-2, 3.0):
        assert device_E(dt, 0.0)[0] == f32(dt)
        assert abs(float(device_dEda(dt, 0.0)) - 0.5 * float(f32(dt)) ** 2) <= 1e-7 * float(f32(dt)) ** 2


@pytest.mark.parametrize("ulps", [0, 2])
def test_dEda_matches_libm(ulps):
    worst = 0.0
    for dt, a in _grid():
        x = abs(float(f32(dt)) * float(f32(a)))
        if x > 30:  # dE/da underflows against E / a there; not a regime of the check
            continue
        got = float(device_dEda(dt, a, ulps))
        want = exact_dEda(dt, a)
        worst = max(worst, abs(got - want) / abs(want))
    assert worst < 2e-5, worst


def test_plain_quotient_fails_the_same_check():
    """The cancelling form (Abar - 1) / a everywhere: at |x| = 1e-6 its error is near 10 %."""
    worst = 0.0
    for dt, a in _grid():
        got, _ = device_E(dt, a, 2, series=False)
        want = exact_E(dt, a)
        worst = max(worst, abs(float(got) - want) / abs(want))
    assert worst > 1e-2


def device_Abar_series(dt, a):
    """Abar as zoh_exact forms it where the series holds: 1 + x phi(x), x = y ln 2, one fmaf at the end."""
    dt, a = f32(dt), f32(a)
    y = f32(dt * f32(a * LOG2E))
    p = fma32(y, PHI3, PHI2)
    p = fma32(p, y, PHI1)
    p = fma32(p, y, f32(1.0))
    return fma32(f32(y * LN2), p, f32(1.0)), y


LN2 = f32(0.6931471805599453)


def test_series_Abar_is_within_an_ulp_of_exp():
    """zoh_exact takes Abar from the series below the threshold (the fp32-output scan and the decode step):
    within one ulp of e^x (of the fp32 x the device forms), where the hardware exp2 is allowed two; its
    errors are also centred, so they do not add up over a long-memory state's thousands of steps."""
    text = open(HEADER).read()
    body = text[text.index("float zoh_exact("):]
    body = body[:body.index("}")]
    assert "fmaf(y * kLn2, phi, 1.0f)" in body and "fabsf(y) < kZohSeriesY" in body
    errs = []
    for dt, a in _grid():
        got, y = device_Abar_series(dt, a)
        if not abs(y) < SERIES_Y:
            continue
        want = math.exp(float(y) * math.log(2.0))
        ulp = float(np.spacing(f32(want)))
        errs.append((float(got) - want) / ulp)
    errs = np.array(errs)
    assert len(errs) > 300
    assert np.abs(errs).max() <= 1.0, np.abs(errs).max()
    assert abs(errs.mean()) < 0.1, errs.mean()
