"""Merged-LoRA weights: plain CPU reference.

TEST INFRASTRUCTURE ONLY (see ``oracle/nvfp4.py``): used by ``tests/`` and
``bench.py``'s CPU legs, never by the product path; it never imports the
product package.

The merged mode folds the LoRA update into the weight before quantising it
(MiniMax-H3 Turbo — one file, no Python, section "What the conversion did",
list "The rest.", item "Backbone": the LoRA's update is merged before
quantizing), as a comparison point for the dynamic path, whose LoRA branch
stays separate (TURBO.md, h3-blackwell-runtime, "Implementation"):

    W' = bf16( W + strength * (alpha / rank) * (B @ A) / s )

with ``W [N, K]``, ``B [N, r]``, ``A [r, K]`` holding bf16 values and ``s``
the per-input-channel ``pre_quant_scale`` (1 when absent).  The base branch
computes ``(x * s) @ W.T`` while the LoRA branch sees the original ``x``
(TURBO.md, "Implementation"), so the folded update carries ``1 / s`` for
``(x * s) @ W'.T`` to reproduce ``x @ (B A).T``.  The sum is
formed in float64 (each product of two bf16 values is exact and r <= 512 terms
of such products lose nothing), then rounded once to bf16, to nearest with
ties to even.  ``W'`` is then packed like any weight (``linear.pack_weight``).
"""
from __future__ import annotations

import numpy as np


def bf16_rne(a) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned
    as float32.  bf16 keeps 8 significant bits: the value is divided by its
    bf16 unit in the last place and rounded half-to-even to an integer.
    Zeros stay zeros; values are assumed finite and inside the normal range."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    nz = a != 0
    f, e = np.frexp(a[nz])                  # a = f * 2^e, 0.5 <= |f| < 1
    ulp = np.ldexp(1.0, e - 8)              # 8 significant bits
    out[nz] = np.round(a[nz] / ulp) * ulp   # np.round: half to even
    return out.astype(np.float32)


def merge_lora(W, A, B, alpha, rank, strength, pre_quant_scale=None) -> np.ndarray:
    """``bf16(W + strength * (alpha/rank) * B @ A / s)`` as float32 [N, K]."""
    W = np.asarray(W, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    c = float(strength) * (float(alpha) / float(rank))
    upd = c * (B @ A)
    if pre_quant_scale is not None:
        upd = upd / np.asarray(pre_quant_scale, dtype=np.float64)[None, :]
    return bf16_rne(W + upd)
