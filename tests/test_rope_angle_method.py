"""Host check of the method behind the kernels' RoPE (cos, sin): the exact fixed-point angle,
the nearest quarter turn taken off in integer arithmetic, and Taylor series of sin (to x^9)
and cos (to x^10) on the remainder |x| <= pi/4, evaluated in fp32 with fused multiply-adds.

The steps are restated here in numpy (fp32 values, each fused multiply-add rounded once from
fp64) and compared with fp64 sin/cos of the same fixed-point angle, over random turn
fractions and position differences and over the quadrant boundaries. The device routine is
exercised through the rotation parity tests (encoded pages, decode and prefill outputs)."""
import numpy as np

F32 = np.float32
M64 = (1 << 64) - 1


def _fma(a, b, c):
    return F32(np.float64(a) * np.float64(b) + np.float64(c))


def _method(delta, turn_frac):
    t = (delta * turn_frac) & M64
    q = ((t + (1 << 61)) & M64) >> 62
    r = (t - (q << 62)) & M64
    r = r - (1 << 64) if r >= 1 << 63 else r           # signed, in [-2^61, 2^61)
    x = F32(F32(r >> 32) * F32(1.46291807926715968e-9))
    x2 = F32(x * x)
    sp = _fma(x2, F32(2.75573192e-6), F32(-1.98412698e-4))
    sp = _fma(x2, sp, F32(8.33333333e-3))
    sp = _fma(x2, sp, F32(-1.66666667e-1))
    sx = _fma(F32(x * x2), sp, x)
    cp = _fma(x2, F32(-2.75573192e-7), F32(2.48015873e-5))
    cp = _fma(x2, cp, F32(-1.38888889e-3))
    cp = _fma(x2, cp, F32(4.16666667e-2))
    cp = _fma(x2, cp, F32(-0.5))
    cx = _fma(x2, cp, F32(1.0))
    cc, ss = (sx, cx) if q & 1 else (cx, sx)
    c = -cc if q in (1, 2) else cc
    s = -ss if q >= 2 else ss
    return float(c), float(s)


def _exact(delta, turn_frac):
    t = (delta * turn_frac) & M64
    ts = t - (1 << 64) if t >= 1 << 63 else t           # turns in [-1/2, 1/2) * 2^64
    a = 2.0 * np.pi * (ts / 2.0 ** 64)
    return np.cos(a), np.sin(a)


def _check(delta, frac, bound=2e-7):
    c, s = _method(delta, frac)
    ce, se = _exact(delta, frac)
    assert abs(c - ce) <= bound and abs(s - se) <= bound, (delta, frac, c, ce, s, se)


def test_random_angles_within_bound():
    rng = np.random.default_rng(7)
    for _ in range(4000):
        frac = int(rng.integers(0, 1 << 63)) * 2 + int(rng.integers(0, 2))
        delta = int(rng.integers(-200000, 200000))
        _check(delta & M64, frac)


def test_quadrant_boundaries_and_special_angles():
    # delta = 1 puts the turn fraction itself on each quarter-turn boundary, +- a few units
    for base in (0, 1 << 61, 1 << 62, 3 << 61, 1 << 63, 5 << 61, 3 << 62, 7 << 61):
        for d in (-(1 << 40), -3, -1, 0, 1, 3, 1 << 40):
            _check(1, (base + d) & M64)
    c, s = _method(0, 12345)                            # zero angle
    assert (c, s) == (1.0, 0.0)
    c, s = _method(1, 1 << 62)                          # a quarter turn
    assert abs(c) < 1e-7 and s == 1.0
    c, s = _method(1, 1 << 63)                          # half a turn
    assert c == -1.0 and abs(s) < 1e-7
