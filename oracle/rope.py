"""Fused Q/K RMSNorm + partial split-half three-axis RoPE: plain CPU reference.

TEST INFRASTRUCTURE ONLY (see ``oracle/nvfp4.py``): used by ``tests/`` and
``bench.py``'s CPU legs, never by the product path; it never imports the
product package.

The step that follows the fused QKV projection (MiniMax-H3 Ultra Fast README,
table "Active optimization stack", row "Attention projections": one fused
in-place Q/K RMSNorm + partial split-half RoPE kernel per block; section
"Kernel path", item 2: three-axis split-half rotary embedding).  The head
size is 128, of which 96 dimensions rotate (MiniMax-H3 Turbo — one file, no
Python: the list of conventions before "Two clocks").  What the pages leave
open is taken in its plainest form:

* ``qkv`` rows are ``[Q | K | V]``, each ``heads * 128`` wide, head-major.
* RMSNorm is per head over its 128 dimensions with a learned gain ``w``
  (one for Q, one for K):  ``y = x / sqrt(mean(x^2) + eps) * w``.
* RoPE then rotates dimensions ``[0, rot)`` of each normalised head, pairing
  ``i`` with ``i + rot/2`` (split-half); the rest pass through.  Pair ``i``
  belongs to axis ``a`` (t, h, w) by concatenation of the axes' pair counts
  ``axis_dims[a] / 2``; inside an axis, pair ``j`` has the frequency
  ``theta ** (-2 j / axis_dims[a])`` and the angle ``pos[a] * freq``:

      out[i]         = y[i] cos(angle_i) - y[i + rot/2] sin(angle_i)
      out[i + rot/2] = y[i + rot/2] cos(angle_i) + y[i] sin(angle_i)

* V is untouched.

Arithmetic in float64; the caller compares against the GPU's bf16 result.
"""
from __future__ import annotations

import numpy as np


def inv_freq(axis_dims=(32, 32, 32), theta=10000.0) -> tuple[np.ndarray, np.ndarray]:
    """Frequencies of the rot/2 pairs and the axis each pair reads its position from."""
    freqs, axes = [], []
    for a, d in enumerate(axis_dims):
        assert d % 2 == 0
        j = np.arange(d // 2, dtype=np.float64)
        freqs.append(float(theta) ** (-2.0 * j / d))
        axes.append(np.full(d // 2, a))
    return np.concatenate(freqs), np.concatenate(axes)


def angles(pos, axis_dims=(32, 32, 32), theta=10000.0) -> np.ndarray:
    """Rotation angle of every (row, pair): ``pos[row, axis(pair)] * freq(pair)``."""
    f, ax = inv_freq(axis_dims, theta)
    pos = np.asarray(pos, dtype=np.float64)
    return pos[:, ax] * f[None, :]


def rms_norm(x, w, eps) -> np.ndarray:
    """Per row of ``x [..., D]``: ``x / sqrt(mean(x^2) + eps) * w``."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * np.asarray(w, dtype=np.float64)


def rope_split_half(y, ang, rot) -> np.ndarray:
    """Rotate dims ``[0, rot)`` of ``y [rows, heads, D]`` by ``ang [rows, rot/2]``."""
    y = np.asarray(y, dtype=np.float64)
    h = rot // 2
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = y[..., :h], y[..., h:rot]
    out = y.copy()
    out[..., :h] = a * c - b * s
    out[..., h:rot] = b * c + a * s
    return out


def qk_norm_rope(qkv, heads, wq, wk, pos, head_dim=128, rot=96, axis_dims=(32, 32, 32), theta=10000.0,
                 eps=1e-6) -> np.ndarray:
    """``qkv [M, 3 * heads * head_dim]`` -> the same layout with Q and K normalised
    and rotated (float64); V copied."""
    qkv = np.asarray(qkv, dtype=np.float64)
    M = qkv.shape[0]
    HD = heads * head_dim
    assert qkv.shape[1] == 3 * HD and sum(axis_dims) == rot and rot % 2 == 0 and rot <= head_dim
    ang = angles(pos, axis_dims, theta)
    out = qkv.copy()
    for part, w in ((0, wq), (1, wk)):
        x = qkv[:, part * HD:(part + 1) * HD].reshape(M, heads, head_dim)
        y = rope_split_half(rms_norm(x, w, eps), ang, rot)
        out[:, part * HD:(part + 1) * HD] = y.reshape(M, HD)
    return out
