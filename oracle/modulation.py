"""Modulation producer (AdaLN shift/scale): plain CPU reference.

TEST INFRASTRUCTURE ONLY (see ``oracle/nvfp4.py``): used by ``tests/`` and
``bench.py``'s CPU legs, never by the product path; it never imports the
product package.

The input of the QKV and gate/up projections is the block's residual stream
normalised and modulated by the AdaLN table: one table row per distinct
timestep, gathered segment-wise over the packed sequence (MiniMax-H3 Ultra
Fast README, "Active optimization stack", row "AdaLN": segment-wise in-place
modulation; MiniMax-H3 AoTI packages: the block gathers from an AdaLN table
with one row per distinct timestep).  The modulation output is the exact BF16
input of the LoRA branch and, after ``pre_quant_scale``, of the NVFP4 packing
(TURBO.md, h3-blackwell-runtime, "Implementation": the modulation producer
packs NVFP4 while it emits the BF16 LoRA input).  Plainest form of what the
pages leave open: LayerNorm without affine parameters over the hidden size,
then ``(1 + scale) * y + shift``:

    y     = (x - mean(x)) / sqrt(var(x) + eps)        (per row, population variance)
    x_mod = bf16( y * (1 + scale[t]) + shift[t] ),    t = row_table[row]

``table[t] = (shift, scale)`` rows of ``K`` values.  Float64 arithmetic, one
bf16 rounding at the end (round to nearest even).
"""
from __future__ import annotations

import numpy as np

from .merged import bf16_rne


def layer_norm(x, eps) -> np.ndarray:
    """Per row of ``x [M, K]``: zero mean, unit (population) variance, no affine."""
    x = np.asarray(x, dtype=np.float64)
    mu = np.mean(x, axis=-1, keepdims=True)
    d = x - mu
    var = np.mean(d * d, axis=-1, keepdims=True)
    return d / np.sqrt(var + float(eps))


def modulate(x, table, row_table, eps=1e-6, round_bf16=True) -> np.ndarray:
    """``x [M, K]``, ``table [T, 2, K]`` (shift, scale), ``row_table [M]`` -> x_mod [M, K]."""
    table = np.asarray(table, dtype=np.float64)
    idx = np.asarray(row_table, dtype=np.int64)
    y = layer_norm(x, eps)
    out = y * (1.0 + table[idx, 1, :]) + table[idx, 0, :]
    return bf16_rne(out) if round_bf16 else out
