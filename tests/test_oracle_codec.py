"""Pins of the NVFP4 codec oracle against things other than itself: the
format's closed-form decoding, torch's independent E4M3 dtype, brute-force
nearest-value search, and the block-scale rule's closed forms."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nvfp4

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------- E2M1
def _e2m1_formula(c):
    """E2M1 from its bit fields: 1 sign, 2 exponent (bias 1), 1 mantissa bit."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def test_e2m1_decode_all_codes():
    got = nvfp4.e2m1_decode(np.arange(16, dtype=np.uint8))
    want = np.array([_e2m1_formula(c) for c in range(16)])
    np.testing.assert_array_equal(got, want)
    # the magnitudes are the NVFP4 element grid
    assert list(want[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_brute(q):
    """Nearest E2M1 magnitude by exhaustive search; ties go to the even code."""
    a = abs(Fraction(float(q)))
    best, best_d = None, None
    for c in range(8):
        d = abs(a - Fraction(_e2m1_formula(c)))
        if best is None or d < best_d or (d == best_d and c % 2 == 0 and best % 2 == 1):
            best, best_d = c, d
    return best | (8 if np.signbit(np.float32(q)) else 0)


def test_e2m1_encode_dense_sweep_vs_bruteforce():
    grid = np.arange(-8.0, 8.0 + 2 ** -12, 2 ** -12, dtype=np.float64).astype(np.float32)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    extra = np.concatenate([ties, -ties, np.nextafter(ties, np.float32(0)), np.nextafter(ties, np.float32(9)),
                            np.array([0.0, -0.0, 6.0, 7.0, 1e30, -1e30, 1e-40, -1e-40], dtype=np.float32)])
    q = np.concatenate([grid, extra]).astype(np.float32)
    got = nvfp4.e2m1_encode(q)
    want = np.array([_e2m1_brute(v) for v in q], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


def test_e2m1_ties_go_to_even_code():
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    want_vals = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    np.testing.assert_array_equal(nvfp4.e2m1_decode(nvfp4.e2m1_encode(ties)), want_vals)
    np.testing.assert_array_equal(nvfp4.e2m1_decode(nvfp4.e2m1_encode(-ties)), [-v for v in want_vals])


def test_e2m1_sign_kept_on_zero():
    assert nvfp4.e2m1_encode(np.float32(-0.1)) == 0x8
    assert nvfp4.e2m1_encode(np.float32(-0.0)) == 0x8
    assert nvfp4.e2m1_encode(np.float32(0.1)) == 0x0
    assert nvfp4.e2m1_encode(np.float32(-100.0)) == 0xF


# ----------------------------------------------------------------------------- E4M3
def _torch_e4m3_decode(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_all_patterns_vs_torch():
    bits = np.arange(256, dtype=np.uint8)
    got = nvfp4.e4m3_decode(bits)
    want = _torch_e4m3_decode(bits)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    assert np.nanmax(got) == 448.0 and np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert got[1] == 2.0 ** -9 and got[8] == 2.0 ** -6


def test_e4m3_encode_vs_torch_in_range():
    rng = np.random.default_rng(123)
    y = np.concatenate([
        rng.uniform(0, 464, 200000).astype(np.float32),
        np.exp2(rng.uniform(-14, 9, 200000)).astype(np.float32),
        nvfp4.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float32),
    ])
    # midpoints between consecutive E4M3 values: exact ties
    vals = nvfp4.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    y = np.concatenate([y, mids]).astype(np.float32)
    y = y[y < 464.0]
    y = np.concatenate([y, -y])
    got = nvfp4.e4m3_encode(y)
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, want)


def test_e4m3_encode_saturates():
    y = np.array([448.0, 463.9, 464.0, 500.0, 1e6, 3e38], dtype=np.float32)
    np.testing.assert_array_equal(nvfp4.e4m3_encode(y), [0x7E] * 6)
    np.testing.assert_array_equal(nvfp4.e4m3_encode(-y), [0xFE] * 6)


def _e4m3_brute(y):
    """Nearest finite non-negative E4M3 value by exhaustive search (ties: even pattern)."""
    best, best_d = None, None
    for b in range(0x7F):
        e, m = b >> 3, b & 7
        val = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        d = abs(Fraction(float(y)) - Fraction(val))
        if best is None or d < best_d or (d == best_d and b % 2 == 0 and best % 2 == 1):
            best, best_d = b, d
    return best


def test_e4m3_encode_vs_bruteforce():
    rng = np.random.default_rng(7)
    y = np.concatenate([np.exp2(rng.uniform(-12, 10, 3000)), rng.uniform(0, 500, 1000)]).astype(np.float32)
    np.testing.assert_array_equal(nvfp4.e4m3_encode(y), [_e4m3_brute(v) for v in y])


# ------------------------------------------------------------------ tensor / block rules
def test_tensor_scale_rule():
    assert nvfp4.tensor_scale(np.float32(2688.0)) == 1.0
    assert nvfp4.tensor_scale(np.float32(0.0)) == 1.0
    assert nvfp4.tensor_scale(np.float32(1e-45)) == 1.0       # quotient underflows to 0
    a = np.float32(12.345)
    assert nvfp4.tensor_scale(a) == np.float32(a / np.float32(2688.0))


@pytest.mark.parametrize("j", [0, 3, 9])
def test_block_scale_closed_form(j):
    """amax = 2688 * 2^-j gives ts = 2^-j exactly; a block whose max is 6 k ts
    (k an exact E4M3 value) gets scale k and its max element code +-6."""
    ts = np.float32(2.0 ** -j)
    ks = nvfp4.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8)).astype(np.float32)
    rows = []
    for k in ks:
        row = np.zeros(16, dtype=np.float32)
        row[3] = np.float32(6.0) * k * ts
        row[7] = -np.float32(0.5) * k * ts
        rows.append(row)
    v = np.stack(rows)
    v[0, 0] = np.float32(2688.0) * ts         # tensor amax element
    amax = nvfp4.tensor_amax(v)
    assert nvfp4.tensor_scale(amax) == ts
    codes, scales = nvfp4.quantize_blocks(v, ts)
    # block 0 holds the tensor amax: scale 448, amax element code 6
    assert scales[0, 0] == 0x7E and codes[0, 0] == 0x7
    for i in range(1, len(ks)):
        assert nvfp4.e4m3_decode(scales[i, 0]) == ks[i]
        assert codes[i, 3] == 0x7                 # +6
        assert codes[i, 7] == 0x9                 # -0.5
        assert np.all(codes[i, [0, 1, 2, 4, 5, 6] + list(range(8, 16))] == 0)


def test_identical_block_values_identical_codes():
    rng = np.random.default_rng(5)
    v = np.repeat(rng.standard_normal((50, 1)).astype(np.float32), 16, axis=1)
    ts = nvfp4.tensor_scale(nvfp4.tensor_amax(v))
    codes, _ = nvfp4.quantize_blocks(v, ts)
    assert np.all(codes == codes[:, :1])
    assert np.all((codes & 7) == 7)               # every element is its block's max -> 6


def test_zero_block_all_zero_codes():
    v = np.zeros((2, 32), dtype=np.float32)
    v[1, 16:] = 3.0
    ts = nvfp4.tensor_scale(nvfp4.tensor_amax(v))
    codes, scales = nvfp4.quantize_blocks(v, ts)
    assert np.all(codes[0] == 0) and np.all(scales[0] == 0) and np.all(codes[1, :16] == 0)


# ------------------------------------------------------------------ brute-force quantise
def _f32_rn(q):
    """The float32 nearest to the exact rational q (ties to the even
    significand), from the binary representation: significand rounded at 24
    bits, or at 2^-149 in the subnormal range.  No float division involved."""
    if q == 0:
        return np.float32(0.0)
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()      # 2^e <= a < 2^(e+2)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    step = Fraction(2) ** max(e - 23, -149)                         # one unit in the last place
    m = round(a / step)                                             # Fraction.__round__: half to even
    val = float(m * step)                                           # exact: at most 25 significant bits
    return np.float32(-val if q < 0 else val)


def test_f32_rn_matches_ieee_division_on_random_pairs():
    # the helper against the IEEE float32 division numpy performs
    rng = np.random.default_rng(21)
    a = (rng.standard_normal(3000) * np.exp2(rng.uniform(-60, 60, 3000))).astype(np.float32)
    b = np.abs(rng.standard_normal(3000) * np.exp2(rng.uniform(-60, 60, 3000))).astype(np.float32) + np.float32(1e-30)
    want = a / b
    got = np.array([_f32_rn(Fraction(float(x)) / Fraction(float(y))) for x, y in zip(a, b)], dtype=np.float32)
    np.testing.assert_array_equal(got, want)


def _quantize_bruteforce(x, s):
    """Element-by-element quantisation with exhaustive nearest-value searches;
    each code from the exact quotient v / d rounded once to float32."""
    M, K = x.shape
    f32 = np.float32
    v = [[f32(x[m, k]) * f32(s[k]) for k in range(K)] for m in range(M)]
    amax = f32(0)
    for m in range(M):
        for k in range(K):
            amax = max(amax, abs(v[m][k]))
    ts = f32(amax) / f32(2688.0)
    if ts == 0:
        ts = f32(1.0)
    codes = np.zeros((M, K), dtype=np.uint8)
    scales = np.zeros((M, K // 16), dtype=np.uint8)
    for m in range(M):
        for b in range(K // 16):
            blk = v[m][16 * b:16 * b + 16]
            bamax = max(abs(t) for t in blk)
            sb = _e4m3_brute(f32(bamax) / (f32(6.0) * ts))
            scales[m, b] = sb
            e, mm = sb >> 3, sb & 7
            sval = (mm / 8.0) * 2.0 ** -6 if e == 0 else (1 + mm / 8.0) * 2.0 ** (e - 7)
            d = f32(sval) * ts
            if d == 0:
                continue
            for i, t in enumerate(blk):
                q = _f32_rn(Fraction(float(t)) / Fraction(float(d)))
                if q == 0 and np.signbit(f32(t)):
                    q = f32(-0.0)
                codes[m, 16 * b + i] = _e2m1_brute(q)
    packed = np.zeros((M, K // 2), dtype=np.uint8)
    for m in range(M):
        for j in range(K // 2):
            packed[m, j] = codes[m, 2 * j] | (codes[m, 2 * j + 1] << 4)
    return packed, scales, ts


def test_codes_follow_the_quotient_where_the_reciprocal_product_differs():
    """Blocks built so that fl(v * fl(1/d)) and fl(v / d) fall on different
    sides of an E2M1 rounding midpoint: quantize_blocks must give the code of
    the exact quotient rounded once (brute force), not the product's."""
    f32 = np.float32
    rng = np.random.default_rng(31)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    ks = nvfp4.e4m3_decode(np.arange(0x30, 0x48, dtype=np.uint8))     # E4M3 values 0.5 .. 4.5
    found = []
    for _ in range(400000):
        k = f32(rng.choice(ks))
        ts = f32(rng.uniform(0.5, 2.0))
        d = f32(k * ts)
        v = f32(f32(rng.choice(mids)) * d)
        for step in range(-3, 4):   # walk v across the midpoint
            vv = v
            for _ in range(abs(step)):
                vv = np.nextafter(vv, f32(np.inf) if step > 0 else f32(0.0))
            if nvfp4.e2m1_encode(vv / d) != nvfp4.e2m1_encode(vv * (f32(1.0) / d)):
                found.append((k, ts, d, vv))
        if len(found) >= 8:
            break
    assert found, "no element whose code depends on the reading"
    for k, ts, d, vv in found:
        row = np.zeros((1, 16), dtype=np.float32)
        row[0, 0] = f32(f32(6.0) * d)             # block max: scale byte k, so the block's d is fl(k * ts)
        row[0, 1] = vv
        row[0, 2] = -vv
        codes, sb = nvfp4.quantize_blocks(row, ts)
        assert nvfp4.e4m3_decode(sb[0, 0]) == k
        for i in (1, 2):
            want = _e2m1_brute(_f32_rn(Fraction(float(row[0, i])) / Fraction(float(d))))
            assert codes[0, i] == want


def test_tiny_blocks_quantise_by_the_quotient():
    """Tensor scales so small that 1/d overflows float32 (d < 2^-128): the
    codes still follow v / d (they are not all zero)."""
    x = np.zeros((2, 32), dtype=np.float32)
    x[0, :16] = np.float32(2.0 ** -130) * np.arange(1, 17, dtype=np.float32)
    x[1, 16:] = -np.float32(2.0 ** -128) * np.arange(16, 0, -1, dtype=np.float32)
    pq, sc, ts = nvfp4.quantize(x, None)
    bq, bsc, bts = _quantize_bruteforce(x, np.ones(32, dtype=np.float32))
    assert ts == bts and ts < 2.0 ** -130
    np.testing.assert_array_equal(sc, bsc)
    np.testing.assert_array_equal(pq, bq)
    d0 = np.float32(nvfp4.e4m3_decode(sc[0, 0])) * ts
    assert d0 < 2.0 ** -128 and not np.isfinite(np.float32(1.0) / d0)
    assert np.any(pq[0, :8] != 0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_quantize_vs_bruteforce_tiny(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    x[1, 5] *= 30.0
    x[2, 16:32] = 0.0
    x[3, 40] = -1e-3
    s = rng.uniform(0.5, 2.0, 64).astype(np.float32)
    pq, sc, ts = nvfp4.quantize(x, s)
    bq, bsc, bts = _quantize_bruteforce(x, s)
    assert ts == bts
    np.testing.assert_array_equal(sc, bsc)
    np.testing.assert_array_equal(pq, bq)


def test_quantize_rows_subset_matches_full():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((300, 128)).astype(np.float32)
    s = rng.uniform(0.5, 2, 128).astype(np.float32)
    pq, sc, ts = nvfp4.quantize(x, s)
    rows = np.array([0, 17, 128, 299])
    pq2, sc2, ts2 = nvfp4.quantize(x, s, rows=rows)
    assert ts == ts2
    np.testing.assert_array_equal(pq[rows], pq2)
    np.testing.assert_array_equal(sc[rows], sc2)
    # chunked amax equals the one-shot amax
    assert nvfp4.tensor_amax_chunked(x, s, chunk_rows=7) == nvfp4.tensor_amax(nvfp4.prescale(x, s))


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(3)
    c = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    p = nvfp4.pack_codes(c)
    assert p[0, 0] == (c[0, 0] | (c[0, 1] << 4))
    np.testing.assert_array_equal(nvfp4.unpack_codes(p), c)


def test_dequantize_small_explicit():
    codes = np.zeros((1, 16), dtype=np.uint8)
    codes[0, :4] = [0x7, 0xF, 0x1, 0x9]
    scales = np.array([[0x38]], dtype=np.uint8)   # E4M3 0x38 = 1.0
    d = nvfp4.dequantize(nvfp4.pack_codes(codes), scales)
    np.testing.assert_array_equal(d[0, :4], [6.0, -6.0, 0.5, -0.5])
    scales2 = np.array([[0x40]], dtype=np.uint8)  # 2.0
    np.testing.assert_array_equal(nvfp4.dequantize(nvfp4.pack_codes(codes), scales2)[0, :2], [12.0, -12.0])
