"""Dynamic-LoRA NVFP4 linear: plain CPU reference of the projection hot path.

TEST INFRASTRUCTURE ONLY (see ``oracle/nvfp4.py``): used by ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline legs, never by the
product path, and it never imports the product package.

Definition followed (TURBO.md, h3-blackwell-runtime, section "Implementation"):

    output = NVFP4_base(x) + strength * (alpha / rank) * B(A(x))

* The NVFP4 base branch quantises ``x * pre_quant_scale``; the BF16 LoRA branch
  receives the ORIGINAL activation ``x`` and is never merged into the packed
  weights (same section, paragraph after the formula).
* Fused QKV uses rank = alpha = 384, the other projections 128 (same place).
* The fused gate/up projection is one matrix ``[gate; up]`` followed by
  ``silu(gate) * up`` (MiniMax-H3 Ultra Fast README, table "Active optimization
  stack", row MLP; section "Kernel path").  LoRA is applied to the linear, i.e.
  before SiLU*up.

Arithmetic: the dequantised operands are exact in float64 and every product is
exact, so the base matmul is the exact sum of the block-scaled products (a
float64 BLAS matmul, error far below the GPU's FP32 accumulation).  The LoRA
branch and SiLU*up are evaluated in float64 as well.
"""
from __future__ import annotations

import numpy as np

from . import nvfp4


def silu_mul(y) -> np.ndarray:
    """``silu(gate) * up`` for ``y = [gate | up]`` split in halves along the last axis."""
    y = np.asarray(y, dtype=np.float64)
    n = y.shape[-1]
    assert n % 2 == 0
    g, u = y[..., : n // 2], y[..., n // 2:]
    return g / (1.0 + np.exp(-g)) * u


def base_matmul(xq, xs, ts_x, wq, ws, ts_w) -> np.ndarray:
    """``ts_x * ts_w * sum_k (e2m1(xq) e4m3(xs)) (e2m1(wq) e4m3(ws))`` in float64."""
    xd = nvfp4.dequantize(xq, xs)          # [M, K]
    wd = nvfp4.dequantize(wq, ws)          # [N, K]
    acc = xd @ wd.T                        # [M, N]
    return float(ts_x) * float(ts_w) * acc


def lora_delta(x, A, B, alpha, rank, strength) -> np.ndarray:
    """``strength * (alpha / rank) * B(A(x))`` in float64 on the original ``x``."""
    x = np.asarray(x, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)    # [r, K]
    B = np.asarray(B, dtype=np.float64)    # [N, r]
    t = x @ A.T                            # [M, r]
    return float(strength) * (float(alpha) / float(rank)) * (t @ B.T)


def forward(x, weight, pre_quant_scale=None, adapter=None, strength=1.0,
            silu_mul_epilogue=False, rows=None, x_amax=None):
    """One projection.

    ``x``        float32 [M, K] holding bf16 values.
    ``weight``   ``(packed codes [N, K/2], scales [N, K/16] row-major, ts_w)``
                 as produced by :func:`pack_weight`.
    ``adapter``  ``None`` or a dict with ``A [r, K]``, ``B [N, r]`` (float32
                 holding bf16 values), ``alpha`` and ``rank``.
    ``rows``     optional row subset to evaluate (the tensor scale of ``x``
                 still comes from the whole tensor, or from ``x_amax``).

    Returns float64 ``[R, N]`` (``[R, N/2]`` with the SiLU*up epilogue).
    """
    x = np.asarray(x, dtype=np.float32)
    xq, xs, ts_x = nvfp4.quantize(x, pre_quant_scale, rows=rows, amax=x_amax)
    wq, ws, ts_w = weight
    y = base_matmul(xq, xs, ts_x, wq, ws, ts_w)
    if adapter is not None and strength != 0.0:
        xr = x if rows is None else x[np.asarray(rows)]
        y = y + lora_delta(xr, adapter["A"], adapter["B"], adapter["alpha"],
                           adapter["rank"], strength)
    if silu_mul_epilogue:
        y = silu_mul(y)
    return y


def pack_weight(w):
    """Quantise a weight ``[N, K]`` once: same rules as activations, ``s = 1``."""
    return nvfp4.quantize(np.asarray(w, dtype=np.float32), None)
