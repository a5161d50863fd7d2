"""Pins of the merged-LoRA oracle (CPU only): bf16 rounding against torch's
own float32 -> bfloat16 conversion and exact rational rounding, the merge
against exact rational arithmetic on a tiny case, and its special cases."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import merged

torch = pytest.importorskip("torch")


def _bf16_values(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).float().numpy()


def _rne_fraction(q: Fraction) -> Fraction:
    """Exact round-to-nearest-even of a positive-or-negative rational to 8
    significant bits."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    # a in [1, 2): 8 significant bits -> unit 2^-7
    m = a * 128
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * Fraction(lo, 128) * (Fraction(2) ** e)


def test_bf16_rne_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000), rng.standard_normal(20000) * 1e-3,
                        rng.standard_normal(20000) * 1e3]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = merged.bf16_rne(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_rne_ties_go_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even mantissa is 1.
    assert merged.bf16_rne(np.array([1.0 + 2.0 ** -8]))[0] == np.float32(1.0)
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    assert merged.bf16_rne(np.array([1.0 + 3 * 2.0 ** -8]))[0] == np.float32(1.0 + 2.0 ** -6)
    assert merged.bf16_rne(np.array([-(1.0 + 2.0 ** -8)]))[0] == np.float32(-1.0)
    assert merged.bf16_rne(np.array([0.0]))[0] == 0.0


def test_bf16_rne_matches_exact_rational_rounding():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(3000) * np.exp(rng.uniform(-20, 20, 3000))
    got = merged.bf16_rne(x)
    for v, g in zip(x, got):
        assert Fraction(float(g)) == _rne_fraction(Fraction(float(v)))


def test_merge_matches_exact_rational_arithmetic():
    rng = np.random.default_rng(2)
    N, K, r = 5, 7, 3
    W = _bf16_values(rng, (N, K), 0.1)
    A = _bf16_values(rng, (r, K), 0.3)
    B = _bf16_values(rng, (N, r), 0.2)
    alpha, strength = 6.0, 0.75
    got = merged.merge_lora(W, A, B, alpha, r, strength)
    c = Fraction(strength) * Fraction(alpha) / r
    for n in range(N):
        for k in range(K):
            s = Fraction(float(W[n, k])) + c * sum(Fraction(float(B[n, j])) * Fraction(float(A[j, k]))
                                                   for j in range(r))
            assert Fraction(float(got[n, k])) == _rne_fraction(s), (n, k)


def test_merge_special_cases():
    rng = np.random.default_rng(3)
    N, K, r = 16, 32, 4
    W = _bf16_values(rng, (N, K), 0.05)
    A = _bf16_values(rng, (r, K))
    B = _bf16_values(rng, (N, r))
    # strength 0: the weight unchanged, bit for bit
    assert np.array_equal(merged.merge_lora(W, A, B, 4.0, r, 0.0), W)
    # zero adapter: unchanged
    assert np.array_equal(merged.merge_lora(W, np.zeros_like(A), B, 4.0, r, 1.0), W)
    # rank-1 unit update touches exactly one element
    A1 = np.zeros((1, K), np.float32)
    B1 = np.zeros((N, 1), np.float32)
    A1[0, 9] = 0.5
    B1[3, 0] = 0.25
    got = merged.merge_lora(W, A1, B1, 1.0, 1, 1.0)
    diff = np.argwhere(got != W)
    assert diff.tolist() in ([[3, 9]], [])
    assert got[3, 9] == merged.bf16_rne(np.array([float(W[3, 9]) + 0.125]))[0]
    # alpha / rank scales the update like strength does
    a = merged.merge_lora(W * 0, A, B, 8.0, r, 0.5)
    b = merged.merge_lora(W * 0, A, B, 4.0, r, 1.0)
    assert np.array_equal(a, b)


def test_merge_divides_the_update_by_the_pre_quant_scale():
    rng = np.random.default_rng(4)
    N, K, r = 6, 8, 2
    W = _bf16_values(rng, (N, K), 0.1)
    A = _bf16_values(rng, (r, K))
    B = _bf16_values(rng, (N, r))
    s = np.array([2.0, 0.5, 1.0, 4.0, 0.25, 1.0, 2.0, 0.5], np.float32)   # powers of two: exact division
    got = merged.merge_lora(W, A, B, 2.0, r, 1.0, s)
    want = merged.merge_lora(W, A / s[None, :], B, 2.0, r, 1.0)
    assert np.array_equal(got, want)
    # without rounding, (x * s) @ W'.T = (x * s) @ W.T + x @ (c B A).T
    x = rng.standard_normal((3, K))
    upd = (1.0 * (B.astype(np.float64) @ A.astype(np.float64))) / s[None, :]
    lhs = (x * s) @ (W.astype(np.float64) + upd).T
    rhs = (x * s) @ W.astype(np.float64).T + x @ (B.astype(np.float64) @ A.astype(np.float64)).T
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
