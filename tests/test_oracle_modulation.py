"""Pins of the modulation-producer oracle (CPU only): LayerNorm closed forms
and invariances, the modulation's special cases (zero table, scale = -1),
the segment gather, and a scalar brute force (math.fsum statistics) on tiny
inputs."""
import math

import numpy as np

from nvfp4_linear_lora_gb300 import synth
from oracle import modulation
from oracle.merged import bf16_rne


def test_layer_norm_closed_forms():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((6, 64)) * 3.0 + 5.0
    eps = 1e-6
    y = modulation.layer_norm(x, eps)
    var = np.var(x, axis=1)
    assert np.allclose(np.mean(y, axis=1), 0.0, atol=1e-13)
    assert np.allclose(np.mean(y * y, axis=1), var / (var + eps), rtol=1e-12)
    # a constant row normalises to zeros
    assert np.array_equal(modulation.layer_norm(np.full((1, 32), 7.0), eps), np.zeros((1, 32)))
    # invariance to a positive affine change of each row (eps = 0)
    a, b = rng.uniform(0.5, 3.0, (6, 1)), rng.standard_normal((6, 1))
    assert np.allclose(modulation.layer_norm(a * x + b, 0.0), modulation.layer_norm(x, 0.0), rtol=1e-11, atol=1e-12)
    # two-point row: values +-1 exactly (eps = 0)
    assert np.allclose(modulation.layer_norm(np.array([[2.0, 4.0, 2.0, 4.0]]), 0.0), [[-1, 1, -1, 1]])


def test_modulation_special_cases():
    rng = np.random.default_rng(1)
    M, K = 10, 48
    x = rng.standard_normal((M, K))
    idx = np.zeros(M, np.int32)
    zero = np.zeros((1, 2, K))
    assert np.array_equal(modulation.modulate(x, zero, idx), bf16_rne(modulation.layer_norm(x, 1e-6)))
    t = np.zeros((1, 2, K)); t[0, 1, :] = -1.0; t[0, 0, :] = 0.375        # (1 + scale) = 0: only the shift
    assert np.array_equal(modulation.modulate(x, t, idx), np.full((M, K), 0.375, np.float32))
    # doubling (1 + scale) doubles the unrounded output
    t = 0.1 * rng.standard_normal((1, 2, K)); t[0, 0, :] = 0.0
    t2 = t.copy(); t2[0, 1, :] = 2 * (1 + t[0, 1, :]) - 1
    a = modulation.modulate(x, t, idx, round_bf16=False)
    b = modulation.modulate(x, t2, idx, round_bf16=False)
    assert np.allclose(b, 2 * a, rtol=1e-13)


def test_segment_gather():
    rng = np.random.default_rng(2)
    K = 16
    x = rng.standard_normal((7, K))
    table = np.zeros((3, 2, K)); table[:, 0, :] = np.array([10.0, 20.0, 30.0])[:, None]   # shift = 10 (t + 1)
    idx = synth.segment_rows((2, 4, 1))
    assert idx.tolist() == [0, 0, 1, 1, 1, 1, 2]
    out = modulation.modulate(x, table, idx, round_bf16=False)
    y = modulation.layer_norm(x, 1e-6)
    for r, t in enumerate(idx):
        assert np.allclose(out[r], y[r] + 10.0 * (t + 1), rtol=1e-14)


def test_brute_force_tiny():
    rng = np.random.default_rng(3)
    M, K, T, eps = 4, 12, 2, 1e-5
    x = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32) * 2 + 1)
    table = 0.2 * rng.standard_normal((T, 2, K))
    idx = np.array([1, 0, 1, 1])
    got = modulation.modulate(x, table, idx, eps)
    for r in range(M):
        vals = [float(v) for v in x[r]]
        mu = math.fsum(vals) / K
        var = math.fsum((v - mu) ** 2 for v in vals) / K
        for k in range(K):
            y = (vals[k] - mu) / math.sqrt(var + eps)
            want = y * (1.0 + table[idx[r], 1, k]) + table[idx[r], 0, k]
            assert got[r, k] == bf16_rne(np.array([want]))[0], (r, k)
