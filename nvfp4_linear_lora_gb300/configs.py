"""The five synthetic workloads of the projection hot path.

Shapes follow the DiT block of the pages: hidden 5120, MLP width 13824, fused
QKV 5120 -> 15360 with LoRA rank/alpha 384, attention-out 5120 -> 5120, fused
gate/up 5120 -> 27648 with SiLU*up, down 13824 -> 5120, all rank/alpha 128
(TURBO.md, h3-blackwell-runtime, "Implementation"; MiniMax-H3 Ultra Fast README,
"Active optimization stack" rows "Attention projections" and "MLP").  The
packed sequence is ragged: S = 37726 for a 16-token prompt, 37728 for an
18-token one (MiniMax-H3 AoTI packages, "What is here").
"""
from __future__ import annotations

HIDDEN = 5120
MLP = 13824

# name, K, N, rank, SiLU*up epilogue
BLOCK_PROJECTIONS = (
    ("qkv", HIDDEN, 3 * HIDDEN, 384, False),
    ("attn_out", HIDDEN, HIDDEN, 128, False),
    ("gate_up", HIDDEN, 2 * MLP, 128, True),
    ("down", MLP, HIDDEN, 128, False),
)

TINY = dict(name="tiny", M=200, K=256, N=384, rank=16, seed=0, law="normal", outlier_frac=0.0)
QKV = dict(name="qkv_9437", M=9437, K=HIDDEN, N=3 * HIDDEN, rank=384, seed=1, law="normal",
           outlier_frac=0.01)
BLOCK_S = 37726
BLOCK_SEED = 2
SWITCH_S = 37728
SWITCH_SEED = 4
SWITCH_ADAPTER_SEEDS = (41, 42)
SWITCH_STRENGTHS = (0.0, 0.5, 1.0)
SWEEP_M = (1024, 4096, 16384, 37726, 65536)

# Q/K RMSNorm + partial split-half three-axis RoPE after the QKV projection:
# 40 heads of 128 (hidden 5120), 96 rotated dimensions (MiniMax-H3 Turbo — one
# file, no Python, list of conventions before "Two clocks"), split equally over
# (t, h, w); positions of a 768 x 1344 canvas in 16-pixel patches (48 x 84 per
# frame) over 9 frames, the rest of the packed rows along t.
ROPE = dict(heads=HIDDEN // 128, head_dim=128, rot=96, axis_dims=(32, 32, 32), theta=10000.0, eps=1e-6,
            frames=9, height=48, width=84)
ROPE_SEED = 8

# Modulation producer: the packed sequence's rows in three segments, each
# gathering its own AdaLN table row (video 9 x 48 x 84 latent patches, then
# the audio and text rows); LayerNorm epsilon 1e-6.
MODULATION = dict(segments=(9 * 48 * 84, 1022, 416), eps=1e-6)
MODULATION_SEED = 9
SWEEP_SEEDS = (3, 4, 5, 6, 7)


def block_flops(S, with_lora=True):
    """Algorithmic FLOPs of the four block projections at sequence length S:
    base ``2 S K N`` plus LoRA ``2 S K r + 2 S r N`` per projection."""
    total = 0
    for _, K, N, r, _ in BLOCK_PROJECTIONS:
        total += 2 * S * K * N
        if with_lora:
            total += 2 * S * K * r + 2 * S * r * N
    return total
