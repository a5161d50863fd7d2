"""Pins of the projection oracle: exact brute force on tiny shapes, the
method's special cases (disabled exactness, pure LoRA, rank-1 closed form,
lossless NVFP4 inputs reducing to a textbook matmul), linearity in strength,
and a quantisation-error sanity band."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import linear, nvfp4

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def _inputs(seed, M, K, N, r):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((M, K)))
    s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    W = _bf16(rng.standard_normal((N, K)) / np.sqrt(K))
    A = _bf16(rng.standard_normal((r, K)) / np.sqrt(K))
    B = _bf16(0.1 * rng.standard_normal((N, r)) / np.sqrt(r))
    return x, s, W, {"A": A, "B": B, "alpha": float(r), "rank": r}


def _dec_e2m1(c):
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return -mag if s else mag


def _dec_e4m3(b):
    e, m = (b >> 3) & 15, b & 7
    return Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def _deq_exact(packed, scales):
    rows, half = packed.shape
    out = []
    for i in range(rows):
        row = []
        for k in range(2 * half):
            byte = int(packed[i, k // 2])
            c = (byte & 15) if k % 2 == 0 else (byte >> 4)
            row.append(_dec_e2m1(c) * _dec_e4m3(int(scales[i, k // 16])))
        out.append(row)
    return out


@pytest.mark.parametrize("M,N", [(1, 1), (3, 2), (4, 3)])
def test_base_matmul_exact_bruteforce(M, N):
    """y[m][n] = ts_x ts_w sum_k xd[m][k] wd[n][k], summed exactly with Fractions."""
    x, s, W, _ = _inputs(10 + M, M, 32, N, 16)
    xq, xs, ts_x = nvfp4.quantize(x, s)
    wq, ws, ts_w = linear.pack_weight(W)
    got = linear.base_matmul(xq, xs, ts_x, wq, ws, ts_w)
    xd, wd = _deq_exact(xq, xs), _deq_exact(wq, ws)
    for m in range(M):
        for n in range(N):
            acc = sum((xd[m][k] * wd[n][k] for k in range(32)), Fraction(0))
            want = Fraction(float(ts_x)) * Fraction(float(ts_w)) * acc
            assert abs(Fraction(got[m, n]) - want) <= abs(want) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


def test_lora_delta_bruteforce():
    M, K, N, r = 3, 32, 2, 16
    x, _, _, ad = _inputs(3, M, K, N, r)
    strength = 0.75
    got = linear.lora_delta(x, ad["A"], ad["B"], ad["alpha"], ad["rank"], strength)
    for m in range(M):
        t = [sum(Fraction(float(ad["A"][j, k])) * Fraction(float(x[m, k])) for k in range(K)) for j in range(r)]
        for n in range(N):
            want = Fraction(strength) * Fraction(ad["alpha"]) / r * sum(Fraction(float(ad["B"][n, j])) * t[j] for j in range(r))
            assert abs(Fraction(got[m, n]) - want) <= abs(want) * Fraction(1, 2 ** 48)


def test_disabled_exactness_bitwise():
    x, s, W, ad = _inputs(1, 40, 64, 48, 16)
    w = linear.pack_weight(W)
    base = linear.forward(x, w, s, adapter=None)
    zero = linear.forward(x, w, s, adapter=ad, strength=0.0)
    assert np.array_equal(base, zero)
    assert not np.array_equal(base, linear.forward(x, w, s, adapter=ad, strength=1.0))


def test_zero_base_weight_is_pure_lora():
    """W = 0: amax 0 -> ts_w = 1, all codes and scales 0, y is the plain LoRA matmul."""
    x, s, W, ad = _inputs(2, 20, 64, 32, 16)
    w = linear.pack_weight(np.zeros_like(W))
    assert w[2] == 1.0 and not w[0].any() and not w[1].any()
    y = linear.forward(x, w, s, adapter=ad, strength=0.5)
    xt, At, Bt = (torch.from_numpy(a).double() for a in (x, ad["A"], ad["B"]))
    want = (0.5 * ad["alpha"] / ad["rank"]) * (xt @ At.T @ Bt.T)
    np.testing.assert_allclose(y, want.numpy(), rtol=1e-12, atol=1e-14)


def test_lora_independent_of_pre_quant_scale():
    x, s, W, ad = _inputs(4, 16, 64, 32, 16)
    w = linear.pack_weight(np.zeros_like(W))
    y1 = linear.forward(x, w, s, adapter=ad)
    y2 = linear.forward(x, w, s * np.float32(3.0), adapter=ad)
    y3 = linear.forward(x, w, None, adapter=ad)
    assert np.array_equal(y1, y2) and np.array_equal(y1, y3)


@pytest.mark.parametrize("which", ["A", "B"])
def test_zero_adapter_factor_gives_base(which):
    x, s, W, ad = _inputs(5, 16, 64, 32, 16)
    w = linear.pack_weight(W)
    ad = dict(ad)
    ad[which] = np.zeros_like(ad[which])
    np.testing.assert_array_equal(linear.forward(x, w, s, adapter=ad), linear.forward(x, w, s))


def test_rank1_adapter_closed_form():
    M, K, N, r = 12, 64, 40, 16
    x, s, W, _ = _inputs(6, M, K, N, r)
    rng = np.random.default_rng(60)
    a = _bf16(rng.standard_normal(K))
    b = _bf16(rng.standard_normal(N))
    A = np.zeros((r, K), np.float32)
    A[0] = a
    B = np.zeros((N, r), np.float32)
    B[:, 0] = b
    ad = {"A": A, "B": B, "alpha": 16.0, "rank": r}
    w = linear.pack_weight(W)
    delta = linear.forward(x, w, s, adapter=ad, strength=0.3) - linear.forward(x, w, s)
    want = 0.3 * (16.0 / r) * np.outer(x.astype(np.float64) @ a.astype(np.float64), b.astype(np.float64))
    np.testing.assert_allclose(delta, want, rtol=1e-9, atol=1e-12)


def _representable(rng, rows, K, ts_exp):
    """A matrix exactly representable in NVFP4 with tensor scale 2^ts_exp:
    each 16-block holds one element +-6 * k * ts (k a power of two, or 448 in
    the block that carries the tensor amax) and E2M1 multiples of k * ts."""
    ts = 2.0 ** ts_exp
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    out = np.zeros((rows, K))
    for i in range(rows):
        for b in range(K // 16):
            k = 2.0 ** rng.integers(-4, 6)
            vals = rng.choice(grid, 16) * rng.choice([-1, 1], 16)
            vals[rng.integers(16)] = 6.0 * rng.choice([-1, 1])
            out[i, 16 * b:16 * b + 16] = vals * k * ts
    out[0, :16] = np.where(np.abs(out[0, :16]) > 0, out[0, :16], 0)
    out[0, 0] = 2688.0 * ts                     # tensor amax: scale 448, code 6
    out[0, 1:16] = np.array([0, 0.5, 1, 1.5, 2, 3, 4, -6, -4, -3, 2, 1, 0.5, 0, 6]) * 448 * ts
    return out.astype(np.float32)


def test_lossless_inputs_reduce_to_plain_matmul():
    rng = np.random.default_rng(8)
    x = _representable(rng, 6, 64, -3)
    W = _representable(rng, 5, 64, -9)
    w = linear.pack_weight(W)
    assert w[2] == np.float32(2.0 ** -9)
    xq, xs, ts_x = nvfp4.quantize(x)
    assert ts_x == np.float32(2.0 ** -3)
    np.testing.assert_array_equal(nvfp4.dequantize(xq, xs) * float(ts_x), x)
    y = linear.forward(x, w, None)
    want = torch.from_numpy(x).double() @ torch.from_numpy(W).double().T
    np.testing.assert_allclose(y, want.numpy(), rtol=1e-13, atol=1e-13)


def test_linear_in_strength():
    x, s, W, ad = _inputs(9, 24, 64, 32, 16)
    w = linear.pack_weight(W)
    y0 = linear.forward(x, w, s, adapter=ad, strength=0.0)
    yh = linear.forward(x, w, s, adapter=ad, strength=0.5)
    y1 = linear.forward(x, w, s, adapter=ad, strength=1.0)
    np.testing.assert_allclose(y1 - y0, 2.0 * (yh - y0), rtol=1e-9, atol=1e-12)


def test_quantisation_error_sanity_band():
    """NVFP4 base vs the unquantised float64 product: a few-% to ~20 % relative
    Frobenius error for Gaussian data.  Pins that scales are applied at all."""
    x, s, W, _ = _inputs(12, 256, 256, 128, 16)
    y = linear.forward(x, linear.pack_weight(W), s)
    ref = (x.astype(np.float64) * s) @ W.astype(np.float64).T
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert 0.02 < rel < 0.25, rel


def test_silu_mul_vs_torch():
    rng = np.random.default_rng(13)
    y = rng.standard_normal((7, 20)) * 4
    g, u = torch.from_numpy(y[:, :10]), torch.from_numpy(y[:, 10:])
    np.testing.assert_allclose(linear.silu_mul(y), (torch.nn.functional.silu(g) * u).numpy(), rtol=1e-14)


def test_gate_up_epilogue_applied_after_lora():
    x, s, W, ad = _inputs(14, 10, 64, 32, 16)
    w = linear.pack_weight(W)
    y = linear.forward(x, w, s, adapter=ad, strength=1.0)
    h = linear.forward(x, w, s, adapter=ad, strength=1.0, silu_mul_epilogue=True)
    np.testing.assert_array_equal(h, linear.silu_mul(y))
    assert h.shape == (10, 16)


def test_row_subset_matches_full():
    x, s, W, ad = _inputs(15, 300, 64, 32, 16)
    w = linear.pack_weight(W)
    full = linear.forward(x, w, s, adapter=ad)
    rows = np.array([0, 5, 127, 128, 299])
    np.testing.assert_array_equal(linear.forward(x, w, s, adapter=ad, rows=rows), full[rows])
