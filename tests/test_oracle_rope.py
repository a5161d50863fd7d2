"""Pins of the Q/K RMSNorm + split-half three-axis RoPE oracle (CPU only).

Closed forms (frequencies, RMSNorm of a constant vector, the rotation of a
one-hot pair), invariants (pair norms, angle 0, relative positions, untouched
V and unrotated dimensions, one axis at a time) and a per-element brute force
on tiny inputs written with scalar math.cos / math.sin."""
import math

import numpy as np

from nvfp4_linear_lora_gb300 import synth
from oracle import rope


def test_inv_freq_closed_form_and_axis_order():
    f, ax = rope.inv_freq((4, 6, 2), theta=10000.0)
    assert np.allclose(f, [1.0, 0.01, 1.0, 10000.0 ** (-2 / 6), 10000.0 ** (-4 / 6), 1.0], rtol=1e-15)
    assert ax.tolist() == [0, 0, 1, 1, 1, 2]


def test_rms_norm_closed_forms():
    D, eps = 128, 1e-6
    for c in (3.0, -0.25, 1e-3):
        y = rope.rms_norm(np.full((1, D), c), np.ones(D), eps)
        assert np.allclose(y, c / math.sqrt(c * c + eps), rtol=1e-14)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, D))
    y = rope.rms_norm(x, np.ones(D), eps)
    ms = np.mean(x * x, axis=1)
    assert np.allclose(np.mean(y * y, axis=1), ms / (ms + eps), rtol=1e-12)
    # scale invariance without eps, and the gain multiplies elementwise
    w = 1 + 0.1 * rng.standard_normal(D)
    assert np.allclose(rope.rms_norm(7.5 * x, w, 0.0), rope.rms_norm(x, w, 0.0), rtol=1e-12)
    assert np.allclose(rope.rms_norm(x, w, eps), y * w, rtol=1e-14)


def test_rotation_of_one_hot_pairs_fixes_the_sign_convention():
    rot, D = 8, 12
    h = rot // 2
    alpha = 0.7
    ang = np.full((1, h), alpha)
    for i in range(h):
        e = np.zeros((1, 1, D)); e[0, 0, i] = 1.0
        out = rope.rope_split_half(e, ang, rot)[0, 0]
        want = np.zeros(D); want[i] = math.cos(alpha); want[i + h] = math.sin(alpha)
        assert np.allclose(out, want, atol=1e-15)
        e = np.zeros((1, 1, D)); e[0, 0, i + h] = 1.0
        out = rope.rope_split_half(e, ang, rot)[0, 0]
        want = np.zeros(D); want[i] = -math.sin(alpha); want[i + h] = math.cos(alpha)
        assert np.allclose(out, want, atol=1e-15)
    e = np.zeros((1, 1, D)); e[0, 0, rot + 1] = 2.0          # beyond rot: untouched
    assert np.array_equal(rope.rope_split_half(e, ang, rot), e)


def test_rotation_invariants():
    rng = np.random.default_rng(1)
    M, H, D, rot = 6, 3, 128, 96
    y = rng.standard_normal((M, H, D))
    ang = rng.uniform(-50, 50, (M, rot // 2))
    out = rope.rope_split_half(y, ang, rot)
    h = rot // 2
    assert np.allclose(out[..., :h] ** 2 + out[..., h:rot] ** 2, y[..., :h] ** 2 + y[..., h:rot] ** 2, rtol=1e-12)
    assert np.array_equal(out[..., rot:], y[..., rot:])
    assert np.allclose(rope.rope_split_half(y, np.zeros_like(ang), rot), y, rtol=0, atol=0)
    # rotating by -angle undoes it
    assert np.allclose(rope.rope_split_half(out, -ang, rot), y, atol=1e-12)


def test_relative_position_property():
    """<rope(q, p1), rope(k, p2)> depends on p1 - p2 only: shifting both
    positions by the same vector leaves every per-head dot product unchanged."""
    rng = np.random.default_rng(2)
    D, rot, dims = 128, 96, (32, 32, 32)
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    p1, p2 = np.array([[3, 10, 41]]), np.array([[1, 7, 2]])
    c = np.array([[5, 11, 23]])
    dot = lambda a, b: float(np.sum(a * b))  # noqa: E731
    d0 = dot(rope.rope_split_half(q, rope.angles(p1, dims), rot), rope.rope_split_half(k, rope.angles(p2, dims), rot))
    d1 = dot(rope.rope_split_half(q, rope.angles(p1 + c, dims), rot),
             rope.rope_split_half(k, rope.angles(p2 + c, dims), rot))
    assert math.isclose(d0, d1, rel_tol=1e-10, abs_tol=1e-10)


def test_one_axis_at_a_time():
    """A position on one axis rotates exactly that axis's pairs."""
    dims = (32, 32, 32)
    for a in range(3):
        pos = np.zeros((1, 3), np.int64); pos[0, a] = 17
        ang = rope.angles(pos, dims)[0]
        nz = np.nonzero(ang)[0]
        lo = 16 * a
        assert nz.min() == lo and nz.max() == lo + 15
        assert math.isclose(ang[lo], 17.0) and math.isclose(ang[lo + 1], 17.0 * 10000.0 ** (-2 / 32))


def test_brute_force_tiny():
    rng = np.random.default_rng(3)
    heads, D, rot, dims, theta, eps = 2, 8, 6, (2, 2, 2), 100.0, 1e-6
    M = 3
    HD = heads * D
    qkv = rng.standard_normal((M, 3 * HD))
    wq, wk = 1 + 0.1 * rng.standard_normal(D), 1 + 0.1 * rng.standard_normal(D)
    pos = np.array([[0, 1, 2], [3, 0, 5], [7, 4, 1]])
    got = rope.qk_norm_rope(qkv, heads, wq, wk, pos, D, rot, dims, theta, eps)
    want = qkv.copy()
    half = rot // 2
    for m in range(M):
        for part, w in ((0, wq), (1, wk)):
            for hh in range(heads):
                base = part * HD + hh * D
                x = [qkv[m, base + d] for d in range(D)]
                inv = 1.0 / math.sqrt(sum(v * v for v in x) / D + eps)
                y = [x[d] * inv * w[d] for d in range(D)]
                for i in range(half):        # pair i: axis i (one pair per axis here), freq theta^0 = 1
                    a = pos[m, i] * 1.0
                    want[m, base + i] = y[i] * math.cos(a) - y[i + half] * math.sin(a)
                    want[m, base + i + half] = y[i + half] * math.cos(a) + y[i] * math.sin(a)
                for d in range(rot, D):
                    want[m, base + d] = y[d]
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
    assert np.array_equal(got[:, 2 * HD:], qkv[:, 2 * HD:])          # V untouched


def test_positions_recipe():
    pos = synth.rope_positions(20, frames=2, height=2, width=3)
    assert pos[:12].tolist() == [[t, h, w] for t in range(2) for h in range(2) for w in range(3)]
    assert pos[12:].tolist() == [[2 + i, 0, 0] for i in range(8)]
