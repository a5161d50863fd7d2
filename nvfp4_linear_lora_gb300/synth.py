"""Seeded synthetic inputs for the projection workloads.

This module only draws random numbers and rounds them to bf16; it holds none
of the method's arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  Generator: numpy PCG64 (``np.random.default_rng(seed)``), whose
streams are identical on x86-64 and aarch64; bf16 rounding is torch's
round-to-nearest-even cast.

Value laws (one per workload, see ``configs.py``):

* activations ``x``: N(0, 1), or Student-t(nu=3); optionally with 1 % of the K
  channels (a seeded permutation) multiplied by 20 ("outlier channels");
* ``pre_quant_scale``: U(0.5, 2) per input channel, float32;
* base weight ``W``: N(0, 1/K), rounded to bf16 before NVFP4 packing;
* LoRA ``A [r, K]``: N(0, 1/K); ``B [N, r]``: 0.1 * N(0, 1/r); both bf16;
* Q/K RMSNorm gains: 1 + 0.1 * N(0, 1); RoPE positions: integer video-grid
  coordinates (``rope_positions``), no randomness;
* residual stream (modulation input): per-row N(0, 1) * U(0.5, 4) + N(0, 1),
  bf16; AdaLN table: 0.1 * N(0, 1) shift and scale per table row; segment
  table: consecutive runs of rows per table row.

Draw order inside one generator: x, outlier channel indices, s, W, A, B.
"""
from __future__ import annotations

import numpy as np
import torch


def bf16_round(a) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returned as float32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def to_bf16_tensor(a) -> torch.Tensor:
    """float32 array holding bf16 values -> torch bf16 CPU tensor (exact)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng, shape, std=1.0, chunk=1 << 24):
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for i in range(0, n, chunk):
        j = min(n, i + chunk)
        out[i:j] = rng.standard_normal(j - i, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out.reshape(shape)


def _student_t(rng, shape, nu, chunk=1 << 22):
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for i in range(0, n, chunk):
        j = min(n, i + chunk)
        out[i:j] = rng.standard_t(nu, j - i).astype(np.float32)
    return out.reshape(shape)


def activation(rng, M, K, law="normal", outlier_frac=0.0, outlier_mult=20.0):
    """x [M, K] as bf16-valued float32 (draws: x, then the outlier channels)."""
    if law == "normal":
        x = _normal(rng, (M, K))
    elif law == "student_t3":
        x = _student_t(rng, (M, K), 3.0)
    else:
        raise ValueError(law)
    if outlier_frac > 0.0:
        n_out = max(1, int(round(outlier_frac * K)))
        idx = rng.permutation(K)[:n_out]
        x[:, idx] *= np.float32(outlier_mult)
    return bf16_round(x)


def pre_quant_scale(rng, K):
    return rng.uniform(0.5, 2.0, K).astype(np.float32)


def weight(rng, N, K):
    return bf16_round(_normal(rng, (N, K), std=1.0 / np.sqrt(K)))


def adapter(rng, N, K, rank, alpha=None):
    A = bf16_round(_normal(rng, (rank, K), std=1.0 / np.sqrt(K)))
    B = bf16_round(_normal(rng, (N, rank), std=0.1 / np.sqrt(rank)))
    return {"A": A, "B": B, "rank": int(rank), "alpha": float(rank if alpha is None else alpha)}


def residual(rng, M, K):
    """A residual-stream stand-in, bf16 [M, K]: per row a N(0, 1) draw scaled by
    U(0.5, 4) and shifted by N(0, 1) (rows with different means and spreads)."""
    g = rng.uniform(0.5, 4.0, (M, 1)).astype(np.float32)
    o = rng.standard_normal((M, 1)).astype(np.float32)
    return bf16_round(_normal(rng, (M, K)) * g + o)


def adaln_table(rng, T, K):
    """AdaLN modulation table, float32 [T, 2, K]: (shift, scale) per distinct
    timestep, both 0.1 * N(0, 1)."""
    return (0.1 * rng.standard_normal((T, 2, K))).astype(np.float32)


def segment_rows(sizes):
    """Table row of every packed row, int32: ``sizes[t]`` consecutive rows use row t."""
    return np.concatenate([np.full(n, t, np.int32) for t, n in enumerate(sizes)])


def norm_gain(rng, D):
    """RMSNorm gain: 1 + 0.1 * N(0, 1) per dimension, float32."""
    return (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)


def rope_positions(M, frames, height, width):
    """Integer (t, h, w) position of every packed row, int32 [M, 3]: a t-major
    frames x height x width video grid first, then the remaining rows along
    t only (t = frames, frames + 1, ...; h = w = 0)."""
    r = np.arange(M, dtype=np.int64)
    grid = frames * height * width
    t = np.where(r < grid, r // (height * width), frames + (r - grid))
    h = np.where(r < grid, (r // width) % height, 0)
    w = np.where(r < grid, r % width, 0)
    return np.stack([t, h, w], axis=1).astype(np.int32)


def projection(seed, M, K, N, rank, law="normal", outlier_frac=0.0, with_adapter=True,
               with_pqs=True):
    """All inputs of one projection from one generator, in the fixed draw order."""
    rng = np.random.default_rng(seed)
    x = activation(rng, M, K, law, outlier_frac)
    s = pre_quant_scale(rng, K) if with_pqs else None
    W = weight(rng, N, K)
    ad = adapter(rng, N, K, rank) if with_adapter else None
    return {"x": x, "pqs": s, "W": W, "adapter": ad, "M": M, "K": K, "N": N, "rank": rank}
