"""The quantising kernels take each element's E2M1 code without a division
per element.  With y = fl(1 / d) they form q_lo = fl(v * fl(y * (1 - 2^-21)))
and q_hi = fl(v * fl(y * (1 + 2^-21))); where both give the same code and
fl(y * (1 + 2^-21)) < 2^100 they take that code, otherwise that element
divides (IEEE float32).  The quantisation rule fixes the code of
the quotient fl(v / d), so the shortcut is exact only if, whenever the two
products agree, the quotient's code agrees with them.

This pins that argument on the CPU in float32 numpy arithmetic over random
values and block scales across the range, over values built to land next to
every E2M1 rounding midpoint, and over tiny and subnormal scales; it also
checks that the bracket has teeth (next to midpoints the single product
fl(v * y) rounds to a different code than the quotient) and stays narrow."""
import numpy as np

from oracle import nvfp4

F32 = np.float32
LO = F32(1.0 - 2.0 ** -21)
HI = F32(1.0 + 2.0 ** -21)
MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=F32)


def _bracket(v, d):
    """The kernels' code step restated: (codes, fast path taken)."""
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        y = F32(1.0) / d
        ylo, yhi = y * LO, y * HI
        clo = nvfp4.e2m1_encode(np.nan_to_num(v * ylo))
        chi = nvfp4.e2m1_encode(np.nan_to_num(v * yhi))
    fast = (yhi < F32(2.0 ** 100)) & (clo == chi)
    return clo, fast


def _check(v, d):
    v = v.astype(F32)
    d = d.astype(F32)
    assert np.all(d > 0)
    want = nvfp4.e2m1_encode(v / d)                  # the rule: code of the IEEE quotient
    clo, fast = _bracket(v, d)
    got = np.where(fast, clo, want)
    assert np.array_equal(got, want), "bracket code differs from the quotient's code"
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        single = nvfp4.e2m1_encode(np.nan_to_num(v * (F32(1.0) / d)))
    return single != want, fast


def test_random_values_and_scales():
    rng = np.random.default_rng(41)
    n = 2_000_000
    d = (2.0 ** rng.uniform(-95, 60, n)).astype(F32)
    q = (rng.standard_normal(n) * 3.0).astype(np.float64)
    v = (q * d.astype(np.float64)).astype(F32)
    _, fast = _check(v, d)
    assert fast.mean() > 0.999


def test_values_next_to_every_e2m1_midpoint():
    rng = np.random.default_rng(42)
    d = (2.0 ** rng.uniform(-30, 30, 4000)).astype(F32)
    m, dd = np.meshgrid(MIDPOINTS, d, indexing="ij")
    base = (m.astype(np.float64) * dd.astype(np.float64)).astype(F32).ravel()
    dd = dd.ravel()
    vs, ds, ks = [], [], []
    for k in range(-12, 13):   # walk v up to 12 ulp either side so the quotient crosses each midpoint
        step = base.copy()
        for _ in range(abs(k)):
            step = np.nextafter(step, F32(np.inf) if k > 0 else F32(0.0))
        vs.append(step)
        ds.append(dd)
        ks.append(np.full(step.size, abs(k)))
    v = np.concatenate(vs)
    d = np.concatenate(ds)
    k = np.concatenate(ks)
    for sign in (1, -1):
        differ, fast = _check(sign * v, d)
        # the bracket has teeth: next to midpoints the single product rounds differently
        assert np.any(differ)
        # and it is narrow (about 2^-21 relative either side): twelve ulp of v
        # away from a midpoint the division is always skipped
        assert np.all(fast[k == 12])


def test_subnormal_values_and_tiny_scales():
    rng = np.random.default_rng(43)
    n = 200_000
    # scales around the fast path's limit 2^-100 and below, values from 0 to 8 d
    d = (2.0 ** rng.uniform(-149, -90, n)).astype(F32)
    d = d[d > 0]
    v = (rng.uniform(-8, 8, d.size) * d.astype(np.float64)).astype(F32)
    _, fast = _check(v, d)
    assert not np.any(fast & (d < F32(2.0 ** -100) * F32(0.999)))
    # subnormal values against normal scales
    d2 = (2.0 ** rng.uniform(-100, -90, n)).astype(F32)
    v2 = (rng.uniform(-1, 1, n) * 2.0 ** -127).astype(F32)
    _check(v2, d2)
    _check(np.array([0.0, -0.0, 1e-45, -1e-45], dtype=F32), np.full(4, 1.0, dtype=F32))


def test_saturation_and_large_quotients():
    d = np.full(6, 0.75, dtype=F32)
    v = np.array([4.5, 4.6, 10.0, -10.0, 1e30, -1e30], dtype=F32)
    _check(v, d)
