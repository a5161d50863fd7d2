"""Host-side arithmetic of the benchmark line (no GPU): the block's FLOP count
and the GEMM's mixed FP4/BF16 roofline, checked against closed forms written
out here from the block's shapes, so that the reported fractions can be
recomputed by hand from the line and the measured peaks.

Shapes: hidden 5120 and MLP width 13824; fused QKV (3 x hidden outputs, LoRA
rank 384), attention out, fused gate/up (2 x MLP outputs, SiLU x up) and down,
rank 128 for the last three (FL2VA Turbo, "Implementation"; MiniMax-H3 Ultra
Fast README, "Active optimization stack")."""
import math

import pytest

pytest.importorskip("torch")
import bench  # noqa: E402


def test_block_flops_closed_form():
    S = 37726
    h, f = 5120, 13824
    # per projection: (K, N, rank)
    shapes = [(h, 3 * h, 384), (h, h, 128), (h, 2 * f, 128), (f, h, 128)]
    base = sum(2 * S * K * N for K, N, _ in shapes)
    down = sum(2 * S * K * r for K, _, r in shapes)
    up = sum(2 * S * r * N for _, N, r in shapes)
    total, b, d, u = bench.block_flops(S)
    assert (b, d, u) == (base, down, up)
    assert total == base + down + up
    # 25.1 TFLOP of projection work per block at this S (the base GEMMs 23.9)
    assert math.isclose(total / 1e12, 25.125, rel_tol=1e-4)
    assert math.isclose(base / 1e12, 23.933, rel_tol=1e-4)


def test_mixed_roofline_closed_form():
    peaks = {"bf16_tflops": 2000.0}
    # 6 TFLOP of FP4 work at 6 x 2000 TF/s takes 0.5 ms; 1 TFLOP of BF16 work 0.5 ms
    r = bench.gemm_roofline(6e12, 1e12, 1.0, peaks)
    assert math.isclose(r["peak"], 7000.0, rel_tol=1e-12)
    assert math.isclose(r["achieved"], 7000.0, rel_tol=1e-12)
    assert math.isclose(r["frac"], 1.0, rel_tol=1e-12)
    # twice the time: half the fraction; no BF16 work: the FP4 peak itself
    assert math.isclose(bench.gemm_roofline(6e12, 1e12, 2.0, peaks)["frac"], 0.5, rel_tol=1e-12)
    assert math.isclose(bench.gemm_roofline(6e12, 0.0, 1.0, peaks)["peak"], 12000.0, rel_tol=1e-12)


def test_whole_job_value_counts_every_rank():
    # weak scaling: N ranks each run one block of F FLOP in the slowest rank's time
    assert math.isclose(bench.whole_job_tflops(25e12, 4, 5.0), 4 * 25e12 / 5e-3 / 1e12, rel_tol=1e-12)
