"""The LoRA branch on its own, on the GPU, against the oracle.

Inside the whole output the LoRA term is only a few percent of the RMS (x
with outlier channels, B ~ 0.1 N(0, 1/r)), so the parity bar on the total
could miss LoRA errors of several percent.  These tests isolate it:

* delta = y(adapter, strength 1) - y(NULL) on the fp32 output mode, element
  by element against the oracle's lora_delta at the parity bar, on the
  CTA-pair kernel at full size (S = 37726 rows; QKV rank 384, the gate/up
  linear rank 128, attention-out rank 128; the tail tile and 512 sampled
  rows);
* zero base weight on the pair kernel: the output is the LoRA term alone
  (with and without SiLU*up), element by element within the bound that the
  branch's bf16 intermediates and FP32 sums allow;
* u = A(x), the bf16 intermediate the amax pass leaves in the workspace,
  against the oracle's t = x A^T within the bf16 rounding plus the FP32
  accumulation bound (rank 384 takes the two-piece MMA path, with its rank
  columns split over CTAs below half a 128-row tile per SM); the
  quantising pass of the MLP's down projection leaves the same u bit for bit,
  and so does a call with few rows, whose tiles split their rank columns
  over several CTAs;
* inputs of tiny magnitude (x ~ 2^-100, W ~ 2^-60 and others), where the
  scaled copy of B would leave the bf16 range and ts_x * ts_w underflows in
  float32: codes stay bit-exact and the output meets the bar."""
import numpy as np
import pytest

from tests._util import assert_parity, have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import configs, h3lin, synth  # noqa: E402
from oracle import linear, nvfp4  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _dev(p, W=None):
    W = p["W"] if W is None else W
    a = p["adapter"]
    return (synth.to_bf16_tensor(p["x"]).cuda(),
            torch.from_numpy(p["pqs"]).cuda() if p["pqs"] is not None else None,
            h3lin.pack_weight(synth.to_bf16_tensor(W).cuda()),
            h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), a["rank"],
                          a["alpha"]))


def _sample_rows(M, seed):
    rng = np.random.default_rng(seed)
    return np.array(sorted(set(range((M - 1) // 128 * 128, M)) | set(rng.choice(M, 512, replace=False).tolist())))


def _lora_ref(p, rows=None):
    a = p["adapter"]
    x = p["x"] if rows is None else p["x"][rows]
    return linear.lora_delta(x, a["A"], a["B"], a["alpha"], a["rank"], 1.0)


def _u_region(ws, M, K, N, r):
    st, off = h3lin.h3lin_forward_workspace_regions(M, K, N, r)
    assert st == h3lin.H3LIN_OK
    return ws[off[2]:off[2] + M * r * 2].view(torch.bfloat16).view(M, r)


# ----------------------------------------------------------- delta, full size
@pytest.mark.parametrize("name,K,N,rank", [("qkv", 5120, 15360, 384), ("gate_up_linear", 5120, 27648, 128),
                                           ("attn_out", 5120, 5120, 128)])
def test_lora_delta_on_the_pair_kernel_at_full_size(name, K, N, rank):
    M = configs.BLOCK_S
    p = synth.projection(7000 + rank + N, M, K, N, rank, outlier_frac=0.01)
    x, s, pw, ad = _dev(p)
    assert N % 256 == 0   # the CTA-pair GEMM
    rows = _sample_rows(M, 17)
    idx = torch.from_numpy(rows).cuda()
    y1 = h3lin.forward(x, pw, s, ad, 1.0, out_dtype=torch.float32).index_select(0, idx)
    y0 = h3lin.forward(x, pw, s, None, 1.0, out_dtype=torch.float32).index_select(0, idx)
    torch.cuda.synchronize()
    delta = (y1.double() - y0.double()).cpu().numpy()
    assert_parity(delta, _lora_ref(p, rows), f"{name}: LoRA delta vs oracle")


# ----------------------------------------------------------- zero base weight
def _lora_elementwise_bound(p, silu):
    """Element-wise bound on |gpu - oracle| for a zero base weight, from the
    branch's bf16 intermediates: u = bf16(t) (t = x A^T accumulated in FP32)
    and B' = bf16(B c') each within 2^-8 relative, FP32 sums over K and over
    the rank, the epilogue's rounding; with SiLU*up the two LoRA halves' errors
    propagate through silu(g) * u (|silu'| <= 1.1) plus the fast exp/divide."""
    a = p["adapter"]
    x, A, B = (np.asarray(v, np.float64) for v in (p["x"], a["A"], a["B"]))
    c = a["alpha"] / a["rank"]
    K, r = A.shape[1], A.shape[0]
    t = x @ A.T
    eu = 2.0 ** -8 * np.abs(t) + 2.0 * K * 2.0 ** -24 * (np.abs(x) @ np.abs(A).T)
    Babs = np.abs(B)
    delta = c * (t @ B.T)
    mag = c * (np.abs(t) @ Babs.T)
    bound = c * (eu @ Babs.T) * (1 + 2.0 ** -8) + 2.0 ** -8 * mag + 2.0 * r * 2.0 ** -24 * mag * 1.01 \
        + 2.0 ** -23 * np.abs(delta)
    if not silu:
        return delta, bound
    n = delta.shape[1] // 2
    g, u, eg, eu2 = delta[:, :n], delta[:, n:], bound[:, :n], bound[:, n:]
    h = linear.silu_mul(delta)
    sg = np.abs(g / (1.0 + np.exp(-g)))
    hb = 1.1 * eg * (np.abs(u) + eu2) + sg * eu2 + 2.0 ** -19 * np.abs(h) + 2.0 ** -30 * np.max(np.abs(h))
    return h, hb


@pytest.mark.parametrize("rank,silu", [(384, False), (128, False), (128, True), (64, True)])
def test_zero_base_weight_on_the_pair_kernel_is_pure_lora(rank, silu):
    M, K, N = 2000, 1024, 2048
    p = synth.projection(8000 + rank + silu, M, K, N, rank, outlier_frac=0.01)
    Wz = np.zeros((N, K), dtype=np.float32)
    x, s, pw, ad = _dev(p, Wz)
    got = h3lin.forward(x, pw, s, ad, 1.0, silu, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    want, bound = _lora_elementwise_bound(p, silu)
    # the oracle's own forward with the zero weight is the LoRA term alone
    ref = linear.forward(p["x"], linear.pack_weight(Wz), p["pqs"], p["adapter"], 1.0, silu)
    np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-300)
    err = np.abs(got - want)
    assert np.all(err <= bound), f"rank {rank} silu {silu}: worst excess {np.max(err - bound):.3e}, " \
                                 f"{np.count_nonzero(err > bound)} elements"
    if not silu:
        assert_parity(got, want, f"pure LoRA rank {rank}")


# ------------------------------------------------------------------- u = A(x)
def _t_bound(x, A):
    t = x.astype(np.float64) @ A.astype(np.float64).T
    acc = np.abs(x.astype(np.float64)) @ np.abs(A.astype(np.float64)).T
    K = x.shape[1]
    return t, 2.0 ** -8 * np.abs(t) + 2.0 * K * 2.0 ** -24 * acc


@pytest.mark.parametrize("M,K,N,rank", [(2000, 5120, 15360, 384), (9437, 5120, 15360, 384), (1537, 5120, 5120, 128),
                                        (300, 1024, 1280, 256), (129, 512, 512, 16)])
def test_u_is_A_of_x_within_bf16_rounding(M, K, N, rank):
    p = synth.projection(9000 + rank, M, K, N, rank, outlier_frac=0.01)
    x, s, pw, ad = _dev(p)
    ws = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(M, K, N, rank))
    h3lin.forward(x, pw, s, ad, 1.0, workspace=ws, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert h3lin.read_status(ws) == 0
    u = _u_region(ws, M, K, N, rank).float().cpu().numpy()
    t, bound = _t_bound(p["x"], p["adapter"]["A"])
    err = np.abs(u - t)
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e}"
    # and it is not trivially satisfied: u carries t to bf16 precision
    assert np.linalg.norm(u - t) / np.linalg.norm(t) < 2.0 ** -8


@pytest.mark.parametrize("rank,M_big,M_small", [(384, 19456, 1000), (128, 19456, 1000)])
def test_u_rows_do_not_depend_on_M(rank, M_big, M_small):
    # the LoRA-down pass picks its work split by M: below half a 128-row tile
    # per SM each tile's rank columns go to several CTAs.  Every u element is
    # still the same sum over K, so the rows of u must come out bit for bit as
    # in a call with enough rows for no split
    K = 1024
    p = synth.projection(9300 + rank, M_big, K, 1536, rank, outlier_frac=0.01)
    x, s, pw, ad = _dev(p)
    us = []
    for M in (M_big, M_small):
        ws = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(M, K, 1536, rank))
        h3lin.forward(x[:M], pw, s, ad, 1.0, workspace=ws, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert h3lin.read_status(ws) == 0
        us.append(_u_region(ws, M, K, 1536, rank).clone())
    assert torch.equal(us[1].view(torch.int16), us[0][:M_small].view(torch.int16))


@pytest.mark.parametrize("M", [700, 30000])
def test_quantising_pass_of_the_mlp_leaves_the_same_u(M):
    # the MLP's down projection computes u = A(h) inside its quantising pass
    # (k_amax_lora with the amax known; from about a 256-row tile per SM on it
    # takes 256-row tiles with two accumulators); the plain chain computes it
    # in the amax pass (128-row tiles): both must leave the same bf16 u
    K, Ngu, Nd, r = 1024, 2048, 1024, 128
    rng = np.random.default_rng(91)
    x = synth.activation(rng, M, K)
    s_gu, s_d = synth.pre_quant_scale(rng, K), synth.pre_quant_scale(rng, Ngu // 2)
    W_gu, W_d = synth.weight(rng, Ngu, K), synth.weight(rng, Nd, Ngu // 2)
    a_gu, a_d = synth.adapter(rng, Ngu, K, r), synth.adapter(rng, Nd, Ngu // 2, r)
    xd = synth.to_bf16_tensor(x).cuda()
    sg, sdn = torch.from_numpy(s_gu).cuda(), torch.from_numpy(s_d).cuda()
    pg, pd = h3lin.pack_weight(synth.to_bf16_tensor(W_gu).cuda()), h3lin.pack_weight(synth.to_bf16_tensor(W_d).cuda())
    ag = h3lin.Adapter(synth.to_bf16_tensor(a_gu["A"]).cuda(), synth.to_bf16_tensor(a_gu["B"]).cuda(), r, a_gu["alpha"])
    an = h3lin.Adapter(synth.to_bf16_tensor(a_d["A"]).cuda(), synth.to_bf16_tensor(a_d["B"]).cuda(), r, a_d["alpha"])
    ws_f = h3lin.new_workspace(h3lin.h3lin_mlp_workspace_bytes(M, K, Ngu, Nd, r))
    h3lin.mlp_forward(xd, pg, pd, sg, sdn, ag, an, workspace=ws_f)
    h = h3lin.forward(xd, pg, sg, ag, 1.0, True)
    ws_c = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(M, Ngu // 2, Nd, r))
    h3lin.forward(h, pd, sdn, an, 1.0, workspace=ws_c)
    torch.cuda.synchronize()
    uf = _u_region(ws_f, M, Ngu // 2, Nd, r)
    uc = _u_region(ws_c, M, Ngu // 2, Nd, r)
    assert torch.equal(uf.view(torch.int16), uc.view(torch.int16))


# ------------------------------------------------------------ tiny magnitudes
TINY_CASES = [
    # x scale, W scale, N (384: single-CTA GEMM, 512: CTA pair), rank, SiLU*up
    (2.0 ** -100, 2.0 ** -60, 384, 64, False),
    (2.0 ** -100, 2.0 ** -60, 512, 64, False),
    (2.0 ** -40, 2.0 ** -60, 512, 32, True),     # SiLU*up: the product stays in float range
    (1.0, 2.0 ** -90, 512, 128, False),
    (2.0 ** -60, 1.0, 512, 128, False),
    (2.0 ** -120, 1.0, 256, 16, False),
]


@pytest.mark.parametrize("xs,wsc,N,rank,silu", TINY_CASES)
def test_tiny_magnitudes_through_the_lora_path(xs, wsc, N, rank, silu):
    M, K = 300, 512
    p = synth.projection(9500 + N + rank, M, K, N, rank, outlier_frac=0.01)
    p["x"] = synth.bf16_round(p["x"] * np.float32(xs))
    p["W"] = synth.bf16_round(p["W"] * np.float32(wsc))
    x, s, pw, ad = _dev(p)
    codes, scales, ts = h3lin.quantize_act(x, s)
    got = h3lin.forward(x, pw, s, ad, 1.0, silu, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rq, rs, rts = nvfp4.quantize(p["x"], p["pqs"])
    assert np.float32(ts.cpu().numpy()[0]) == rts
    assert np.array_equal(codes.cpu().numpy(), rq)
    out = got.cpu().numpy()
    assert np.all(np.isfinite(out))
    ref = linear.forward(p["x"], linear.pack_weight(p["W"]), p["pqs"], p["adapter"], 1.0, silu)
    if not silu:
        assert_parity(out, ref, f"x*{xs:g} W*{wsc:g} N={N} r={rank}")
        return
    # SiLU*up: the tiny weight leaves a base term 2^-60 below the LoRA one, so
    # the output is the LoRA term's (heavy-tailed) silu(g) * u: element-wise
    # bound of the bf16 LoRA intermediates, plus twice the base term's size
    lora_h, bound = _lora_elementwise_bound(p, True)
    base = np.abs(ref - lora_h)
    assert np.max(base) <= 2.0 ** -40 * np.max(np.abs(ref))
    err = np.abs(out.astype(np.float64) - ref)
    assert np.all(err <= bound + 2.0 * base), f"worst excess {np.max(err - bound - 2 * base):.3e}"
