"""The QKV projection with Q/K RMSNorm + split-half RoPE in its GEMM epilogue
(h3lin_forward_qk_rope) on the GPU.

Its epilogue computes every Q and K value with the same float operations as
the separate in-place step applied to the stored bf16 projection, so the
fused output must equal h3lin_forward followed by h3lin_qk_norm_rope bit for
bit (V included), on the full QKV shape (S = 37726, 40 heads, rank 384) as on
small ragged shapes, for tiny tensor scales (the two-factor epilogue scale)
and with eps = 0.  Against the oracle: sampled rows of the fused output meet
the parity bar against the oracle's RMSNorm + RoPE of its own projection."""
import numpy as np
import pytest

from tests._util import assert_parity, have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import configs, h3lin, synth  # noqa: E402
from oracle import linear, rope  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _inputs(seed, M, K, heads, rank, x_mul=1.0, w_mul=1.0, grid=(3, 5, 7)):
    N = 3 * heads * 128
    p = synth.projection(seed, M, K, N, rank, outlier_frac=0.01, with_adapter=rank > 0)
    rng = np.random.default_rng(seed + 1)
    x = synth.bf16_round(p["x"] * x_mul)
    W = synth.bf16_round(p["W"] * w_mul)
    dev = dict(x=synth.to_bf16_tensor(x).cuda(), pqs=torch.from_numpy(p["pqs"]).cuda(),
               pw=h3lin.pack_weight(synth.to_bf16_tensor(W).cuda()),
               qg=torch.from_numpy(synth.norm_gain(rng, 128)).cuda(),
               kg=torch.from_numpy(synth.norm_gain(rng, 128)).cuda(),
               pos=torch.from_numpy(synth.rope_positions(M, *grid)).cuda())
    if rank:
        a = p["adapter"]
        dev["ad"] = h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(),
                                  a["rank"], a["alpha"])
    else:
        dev["ad"] = None
    host = dict(p, x=x, W=W)
    return host, dev


def _two_step(d, heads, strength, eps):
    y = h3lin.forward(d["x"], d["pw"], d["pqs"], d["ad"], strength)
    return h3lin.qk_norm_rope(y, d["qg"], d["kg"], d["pos"], heads, eps=eps)


def _fused(d, heads, strength, eps):
    M, K = d["x"].shape
    ws = h3lin.new_workspace(h3lin.h3lin_forward_qk_rope_workspace_bytes(M, K, d["pw"].N,
                                                                        d["ad"].rank if d["ad"] else 0))
    out = h3lin.forward_qk_rope(d["x"], d["pw"], d["qg"], d["kg"], d["pos"], heads, d["pqs"], d["ad"], strength,
                                eps=eps, workspace=ws)
    torch.cuda.synchronize()
    assert h3lin.read_status(ws) == 0
    return out


def _assert_bits_equal(got, want, what):
    g = got.view(torch.int16)
    w = want.view(torch.int16)
    if not torch.equal(g, w):
        bad = (g != w).nonzero()
        raise AssertionError(f"{what}: {bad.shape[0]} elements differ, first at {bad[0].tolist()}")


@pytest.mark.parametrize("M,K,heads,rank,strength,eps", [
    (300, 512, 4, 32, 1.0, 1e-6),      # ragged rows, Q/K/V tiles, LoRA
    (1, 256, 2, 0, 1.0, 1e-6),         # one row, base only
    (513, 1024, 6, 384, 0.5, 1e-6),    # rank 384 (two-piece A(x)), strength 0.5
    (700, 512, 2, 16, 1.0, 0.0),       # eps = 0
    (257, 768, 8, 128, 0.0, 1e-5),     # strength 0: the base path
])
def test_fused_equals_forward_then_qk_norm_rope(M, K, heads, rank, strength, eps):
    _, d = _inputs(100 + M + heads, M, K, heads, rank)
    want = _two_step(d, heads, strength, eps)
    got = _fused(d, heads, strength, eps)
    _assert_bits_equal(got, want, f"M={M} K={K} heads={heads} rank={rank}")


def test_fused_with_tiny_tensor_scales():
    # x ~ 2^-40, W ~ 2^-60: ts_x * ts_w underflows in float32, so the epilogue
    # scale is applied as two factors; the fused epilogue must do the same
    M, K, heads, rank = 260, 512, 4, 32
    _, d = _inputs(77, M, K, heads, rank, x_mul=2.0 ** -40, w_mul=2.0 ** -60)
    want = _two_step(d, heads, 1.0, 1e-30)
    got = _fused(d, heads, 1.0, 1e-30)
    assert torch.isfinite(got.float()).all()
    _assert_bits_equal(got, want, "tiny tensor scales")


def test_fused_equals_two_step_on_the_block_qkv_shape():
    S, K, heads, rank = configs.BLOCK_S, configs.HIDDEN, configs.ROPE["heads"], 384
    c = configs.ROPE
    _, d = _inputs(4242, S, K, heads, rank, grid=(c["frames"], c["height"], c["width"]))
    want = _two_step(d, heads, 1.0, c["eps"])
    got = _fused(d, heads, 1.0, c["eps"])
    _assert_bits_equal(got, want, "S=37726 QKV")


def test_fused_rows_against_the_oracle():
    M, K, heads, rank = 400, 512, 4, 32
    host, d = _inputs(55, M, K, heads, rank)
    got = _fused(d, heads, 1.0, 1e-6).float().cpu().numpy().astype(np.float64)
    rows = np.array(sorted(set(range(M - 20, M)) | set(np.random.default_rng(3).choice(M, 60, replace=False))))
    y = linear.forward(host["x"], linear.pack_weight(host["W"]), host["pqs"], host["adapter"], 1.0, False, rows=rows)
    qkv = synth.bf16_round(y)   # the projection as stored (bf16), then the step
    pos = synth.rope_positions(M, 3, 5, 7)[rows]
    ref = rope.qk_norm_rope(qkv, heads, d["qg"].cpu().numpy(), d["kg"].cpu().numpy(), pos, 128, 96, (32, 32, 32),
                            10000.0, 1e-6)
    HD = heads * 128
    assert_parity(got[rows, :2 * HD], ref[:, :2 * HD], "fused Q/K vs oracle")
    assert_parity(got[rows, 2 * HD:], ref[:, 2 * HD:], "fused V vs oracle")
