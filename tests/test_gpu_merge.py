"""Merged-LoRA comparison mode on the GPU against the oracle:
h3lin_merge_lora's W' within one bf16 unit of the exact merge (FP32
accumulation vs exact rounding), in place or not, strength 0 bit-identical;
the merged weight packed bit-exactly and its base-only forward at the parity
bar against the oracle's forward on the same merged weight."""
import numpy as np
import pytest

from tests._util import assert_parity, have_gpu, native_to_rowmajor

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import h3lin, synth  # noqa: E402
from oracle import linear, merged  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _bf16_ulp(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(v == 0, 1.0, v))
    return np.ldexp(1.0, e - 8)


def _dev_adapter(a):
    return h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(),
                         a["rank"], a["alpha"])


MERGE_CASES = [
    # N, K, rank, alpha, strength, with pre_quant_scale
    (384, 256, 16, 16.0, 1.0, False),
    (200, 320, 48, 96.0, 0.5, True),
    (1280, 1024, 128, 128.0, 1.0, True),
    (515, 5120, 384, 384.0, 0.75, True),
]


@pytest.mark.parametrize("N,K,rank,alpha,strength,with_s", MERGE_CASES)
def test_merge_matches_oracle(N, K, rank, alpha, strength, with_s):
    p = synth.projection(500 + N + K + rank, 8, K, N, rank)
    a = dict(p["adapter"], alpha=alpha)
    W = synth.to_bf16_tensor(p["W"]).cuda()
    s_host = p["pqs"] if with_s else None
    s_dev = torch.from_numpy(p["pqs"]).cuda() if with_s else None
    got = h3lin.merge_lora(W, _dev_adapter(a), strength, s_dev).float().cpu().numpy()
    want = merged.merge_lora(p["W"], a["A"], a["B"], alpha, rank, strength, s_host)
    diff = np.abs(got.astype(np.float64) - want.astype(np.float64))
    # one bf16 unit for the two roundings, plus the FP32 accumulation bound
    # (rank + 4) * 2^-24 * (|W| + |c| |B| @ |A| / s): where W and the update
    # cancel, the latter dominates the tiny result
    c = strength * alpha / rank
    inv_s = 1.0 / np.asarray(s_host, np.float64)[None, :] if with_s else 1.0
    acc_bound = (rank + 4) * 2.0 ** -24 * (np.abs(p["W"]).astype(np.float64)
                                            + abs(c) * (np.abs(a["B"]).astype(np.float64)
                                                        @ np.abs(a["A"]).astype(np.float64)) * inv_s)
    assert np.all(diff <= _bf16_ulp(want) + acc_bound), f"max excess {(diff - _bf16_ulp(want) - acc_bound).max():.3e}"
    assert np.mean(diff == 0) >= 0.999, f"exact fraction {np.mean(diff == 0):.5f}"
    # in place gives the same bits
    W2 = W.clone()
    h3lin.merge_lora(W2, _dev_adapter(a), strength, s_dev, out=W2)
    assert torch.equal(W2.cpu(), torch.from_numpy(got).to(torch.bfloat16))


def test_merge_strength_zero_is_identity():
    p = synth.projection(77, 8, 512, 256, 64)
    W = synth.to_bf16_tensor(p["W"]).cuda()
    got = h3lin.merge_lora(W, _dev_adapter(p["adapter"]), 0.0)
    assert torch.equal(got, W)


@pytest.mark.parametrize("M,K,N,rank,silu", [(300, 1024, 1280, 128, False), (257, 512, 512, 64, True)])
def test_merged_forward_matches_oracle(M, K, N, rank, silu):
    p = synth.projection(900 + M + N, M, K, N, rank, outlier_frac=0.01)
    a = p["adapter"]
    W = synth.to_bf16_tensor(p["W"]).cuda()
    s = torch.from_numpy(p["pqs"]).cuda()
    Wm = h3lin.merge_lora(W, _dev_adapter(a), 1.0, s)
    pw = h3lin.pack_weight(Wm)
    Wm_host = Wm.float().cpu().numpy()
    # the packed merged weight is bit-exact against the oracle's packing of the same bf16 values
    rq, rs, rts = linear.pack_weight(Wm_host)
    assert np.array_equal(pw.codes.cpu().numpy(), rq)
    np.testing.assert_array_equal(native_to_rowmajor(pw.scales.cpu().numpy(), N, K), rs)
    assert np.float32(pw.tensor_scale.cpu().numpy()[0]) == rts
    x = synth.to_bf16_tensor(p["x"]).cuda()
    y = h3lin.forward(x, pw, s, None, 1.0, silu_mul=silu, out_dtype=torch.float32).cpu().numpy()
    ref = linear.forward(p["x"], (rq, rs, rts), p["pqs"], None, 1.0, silu)
    assert_parity(y, ref, f"merged M={M} K={K} N={N} r={rank} silu={silu}")
    # merged vs dynamic: both carry FP4 noise of differently quantised weights, so
    # each is compared with the exact unquantised result and the merged path's
    # error must stay of the same size as the dynamic path's
    xd = np.asarray(p["x"], np.float64)
    xs = xd * np.asarray(p["pqs"], np.float64)[None, :]        # the base branch sees x * pre_quant_scale
    exact = xs @ np.asarray(p["W"], np.float64).T + (xd @ np.asarray(a["A"], np.float64).T) @ np.asarray(a["B"], np.float64).T
    if silu:
        exact = linear.silu_mul(exact)
    dyn = linear.forward(p["x"], linear.pack_weight(p["W"]), p["pqs"], a, 1.0, silu)
    e_m = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    e_d = np.linalg.norm(dyn - exact) / np.linalg.norm(exact)
    assert e_m <= 1.5 * e_d + 0.01, f"merged {e_m:.3e} vs dynamic {e_d:.3e} (rel. Frobenius to exact)"
