"""The quotient the e4m3 kernels use in place of an IEEE division (Markstein's
method: r = RN(1/d), q = RN(v r), q' = RN(q + RN(v - q d) r) with both
corrections as FMAs), emulated exactly in float64 on the CPU and compared
with numpy's IEEE FP32 division for bf16 v.

Within the band the kernels use it in (|q| in [2^-20, 1024), |d| in
[2^-60, 2^60]) exponents only scale every step, so v and d in [1, 2) cover
all cases: all 128 bf16 significands of v times every STRIDE-th of the 2^23
significands of d (STRIDE = 1 with MH3_FULL_DIVISION_CHECK=1: about
2.5 minutes; the default stride takes a few seconds)."""
import os

import numpy as np

STRIDE = 1 if os.environ.get("MH3_FULL_DIVISION_CHECK") == "1" else 61


def _rn32_of_sum(s, t):
    """RN32(s + t) where s = fl64(s + t) and t its exact error (TwoSum):
    float64 keeps 29 more bits, so only a float32 midpoint s with t != 0
    needs t's sign to pick the neighbour."""
    f = s.astype(np.float32)
    back = f.astype(np.float64)
    up = np.nextafter(f, np.float32(np.inf))
    dn = np.nextafter(f, np.float32(-np.inf))
    mid_up = (back + up.astype(np.float64)) / 2
    mid_dn = (back + dn.astype(np.float64)) / 2
    out = f.copy()
    sel = (s == mid_up) & (t > 0)
    out[sel] = up[sel]
    sel = (s == mid_dn) & (t < 0)
    out[sel] = dn[sel]
    return out


def fma32(a, b, c):
    a, b, c = (x.astype(np.float64) for x in (a, b, c))
    p = a * b  # exact: 24 x 24 significand bits
    s = p + c
    bb = s - p
    t = (p - (s - bb)) + (c - bb)
    return _rn32_of_sum(s, t)


def markstein(v, d):
    r = (np.float32(1.0) / d).astype(np.float32)
    q = (v * r).astype(np.float32)
    return fma32(fma32(-q, d, v), r, q)


def test_fma_emulation_against_exact_rationals():
    from fractions import Fraction
    rng = np.random.default_rng(0)
    n = 3000
    a = rng.standard_normal(n).astype(np.float32)
    b = rng.standard_normal(n).astype(np.float32)
    c = -(a * b).astype(np.float32) * (1 + rng.integers(-3, 4, n) * 2.0 ** -23).astype(np.float32)
    c = np.concatenate([c, rng.standard_normal(n).astype(np.float32) * 1e-3]).astype(np.float32)
    a, b = np.concatenate([a, a]), np.concatenate([b, b])
    got = fma32(a, b, c)

    def rn32(x):
        f = np.float32(float(x))
        cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
        return min(cands, key=lambda y: (abs(Fraction(float(y)) - x),
                                         int(np.array(y).view(np.uint32)) & 1))

    for i in range(a.size):
        exact = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        assert rn32(exact) == got[i], i
    # a product exactly on a float32 midpoint, nudged either way
    m = np.float32(1 + 2.0 ** -12)
    tie = fma32(np.full(3, m), np.full(3, m), np.array([0, 2.0 ** -60, -2.0 ** -60], np.float32))
    assert tie[0] == np.float32(1 + 2.0 ** -11) and tie[1] > tie[0] and tie[2] == tie[0]


def test_markstein_quotient_equals_ieee_division():
    vs = (1.0 + np.arange(128, dtype=np.float32) / 128).astype(np.float32)
    for start in range(0, 1 << 23, 1 << 18):
        m = np.arange(start, min(start + (1 << 18), 1 << 23), STRIDE, dtype=np.uint32)
        ds = (np.uint32(0x3F800000) | m).view(np.float32)
        V = np.repeat(vs, ds.size)
        D = np.tile(ds, vs.size)
        got = markstein(V, D)
        ref = (V / D).astype(np.float32)
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (V[bad[0]], D[bad[0]], got[bad[0]], ref[bad[0]])


def test_markstein_division_by_six_for_every_bf16_value():
    """The NVFP4 block scale's RN(amax / 6) on the GPU: the Markstein quotient
    with the constant r = RN(1/6), used for amax in [2^-100, 2^127) (outside,
    a true division).  Every positive bf16 value in that range."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)          # positive finite bf16
    v = (bits << 16).view(np.float32)
    v = v[(v >= np.float32(2.0 ** -100)) & (v < np.float32(2.0 ** 127))]
    d = np.full(v.shape, 6.0, dtype=np.float32)
    got = markstein(v, d)
    ref = (v / d).astype(np.float32)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (v[bad[0]], got[bad[0]], ref[bad[0]])
