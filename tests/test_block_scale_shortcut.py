"""The quantising kernels take a block's scale byte without a division per
block: they round p = fl(bm * fl(1 / fl(6 ts))) to E4M3, and take the IEEE
quotient fl(bm / fl(6 ts)) only when p lies within 3 ulp of an E4M3 rounding
midpoint or below 2^-6.  The quantisation rule fixes the quotient (block
scale = E4M3_sat(bamax / (6 ts)), float32, round to nearest even), so the
shortcut is exact only if both values always round to the same E4M3 byte.

This pins that argument on the CPU, in float32 numpy arithmetic, over random
block maxima and tensor scales across the whole range and over values built
to land next to every E4M3 midpoint; it also checks that the fallback window
is needed (without it, some bytes differ) and is never missed."""
import numpy as np

from oracle import nvfp4

F32 = np.float32


def _shortcut(bm, six_ts):
    """The kernels' block-scale step restated: (bytes, fallback taken)."""
    p = bm * (F32(1.0) / six_ts)
    low = p.view(np.uint32) & np.uint32(0xFFFFF)
    near = (low - np.uint32(0x80000 - 3)) <= np.uint32(6)   # unsigned wrap
    fallback = (p < F32(2.0 ** -6)) | near
    return p, fallback


def _check(bm, six_ts):
    bm = bm.astype(F32)
    six_ts = six_ts.astype(F32)
    q = bm / six_ts                                   # the rule's IEEE quotient
    p, fallback = _shortcut(bm, six_ts)
    want = nvfp4.e4m3_encode(q)
    fast = nvfp4.e4m3_encode(p)
    got = np.where(fallback, want, fast)
    assert np.array_equal(got, want)
    return fast != want, fallback


def test_random_block_maxima_and_tensor_scales():
    rng = np.random.default_rng(11)
    n = 400_000
    ts = (2.0 ** rng.uniform(-20, 10, n)).astype(F32)
    six_ts = F32(6.0) * ts
    # block maxima from 1/1e6 of the tensor's largest scale to the largest (ratio <= 448)
    ratio = (2.0 ** rng.uniform(-20, np.log2(448.0), n)).astype(F32)
    bm = (ratio.astype(np.float64) * six_ts.astype(np.float64)).astype(F32)
    differ, fallback = _check(bm, six_ts)
    assert not np.any(differ & ~fallback)


def test_values_next_to_every_e4m3_midpoint():
    # every rounding midpoint between consecutive normal E4M3 values up to 448
    vals = np.sort(np.abs(nvfp4.e4m3_decode(np.arange(0x08, 0x7F, dtype=np.uint8))))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(F32)
    rng = np.random.default_rng(12)
    six_ts = (6.0 * 2.0 ** rng.uniform(-12, 6, 64)).astype(F32)
    m, s = np.meshgrid(mids, six_ts, indexing="ij")
    base = (m.astype(np.float64) * s.astype(np.float64)).astype(F32).ravel()
    s = s.ravel()
    bms, sts = [], []
    for k in range(-12, 13):   # walk bm up to 12 ulp either side so p crosses each midpoint
        step = base.copy()
        for _ in range(abs(k)):
            step = np.nextafter(step, F32(np.inf) if k > 0 else F32(0.0))
        bms.append(step)
        sts.append(s)
    bm = np.concatenate(bms).astype(F32)
    st = np.concatenate(sts).astype(F32)
    differ, fallback = _check(bm, st)
    # the window has teeth: next to midpoints the product alone rounds differently
    assert np.any(differ)
    assert not np.any(differ & ~fallback)
    # and it stays narrow: most of these near-midpoint cases still skip the division
    assert fallback.mean() < 0.5


def test_subnormal_e4m3_range_and_zero_take_the_division():
    six_ts = np.full(7, 6.0, dtype=F32)
    bm = np.array([0.0, 1e-30, 6 * 2.0 ** -10, 6 * 2.0 ** -9 * 1.5, 6 * 2.0 ** -7, 6 * 2.0 ** -6 * 0.999, 6 * 2.0 ** -6],
                  dtype=F32)
    _, fallback = _check(bm, six_ts)
    assert np.all(fallback[:-1]) and not fallback[-1]
