"""GPU parity of h3lin_forward against the oracle at sizes the oracle finishes
in seconds: several tiles, ragged M tails, every epilogue/adapter mode, plus
the method's exactness and switching properties.

Floating-point parity is judged on the fp32 output mode (the epilogue value
before the output cast); the bf16 output is then checked to be exactly the
round-to-nearest-even of that fp32 value, so the bf16 store adds nothing but
its own rounding."""
import numpy as np
import pytest

from tests._util import assert_parity, have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import configs, h3lin, synth  # noqa: E402
from oracle import linear  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def to_dev(p):
    d = {"x": synth.to_bf16_tensor(p["x"]).cuda(),
         "pqs": torch.from_numpy(p["pqs"]).cuda() if p["pqs"] is not None else None,
         "W": synth.to_bf16_tensor(p["W"]).cuda()}
    ad = p["adapter"]
    d["adapter"] = None if ad is None else h3lin.Adapter(synth.to_bf16_tensor(ad["A"]).cuda(),
                                                         synth.to_bf16_tensor(ad["B"]).cuda(), ad["rank"], ad["alpha"])
    return d


def run(p, strength=1.0, silu=False, use_adapter=True, dev=None, pw=None, out_dtype=torch.float32):
    dev = dev or to_dev(p)
    pw = pw or h3lin.pack_weight(dev["W"])
    out = h3lin.forward(dev["x"], pw, dev["pqs"], dev["adapter"] if use_adapter else None, strength, silu,
                        out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), dev, pw


def assert_bf16_is_rounded_f32(p, strength=1.0, silu=False, use_adapter=True, dev=None, pw=None):
    f32, dev, pw = run(p, strength, silu, use_adapter, dev, pw, torch.float32)
    b16, _, _ = run(p, strength, silu, use_adapter, dev, pw, torch.bfloat16)
    want = torch.from_numpy(f32).to(torch.bfloat16).float().numpy()
    assert np.array_equal(b16.view(np.uint32), want.view(np.uint32))


def ref(p, strength=1.0, silu=False, use_adapter=True):
    return linear.forward(p["x"], linear.pack_weight(p["W"]), p["pqs"], p["adapter"] if use_adapter else None,
                          strength, silu)


CASES = [
    # M, K, N, rank, silu
    (200, 256, 384, 16, False),      # the tiny single-projection workload
    (1, 64, 128, 16, False),
    (129, 320, 256, 32, False),
    (300, 256, 512, 64, True),
    (130, 128, 256, 128, True),
    (257, 512, 384, 384, False),
    (64, 1024, 768, 256, False),
    (384, 256, 256, 288, False),
    (1000, 1024, 1280, 128, False),
]


@pytest.mark.parametrize("M,K,N,rank,silu", CASES)
def test_forward_matches_oracle(M, K, N, rank, silu):
    p = synth.projection(1000 + M + K + N + rank, M, K, N, rank, outlier_frac=0.01)
    got, dev, pw = run(p, silu=silu)
    assert got.shape == (M, N // 2 if silu else N)
    assert_parity(got, ref(p, silu=silu), f"M={M} K={K} N={N} r={rank} silu={silu}")
    assert_bf16_is_rounded_f32(p, silu=silu, dev=dev, pw=pw)


@pytest.mark.parametrize("M,K,N,rank,silu", CASES[:6])
def test_base_path_matches_oracle(M, K, N, rank, silu):
    p = synth.projection(2000 + M, M, K, N, rank)
    got, dev, pw = run(p, silu=silu, use_adapter=False)
    assert_parity(got, ref(p, silu=silu, use_adapter=False), "base")
    assert_bf16_is_rounded_f32(p, silu=silu, use_adapter=False, dev=dev, pw=pw)


# CTA-pair GEMM (N % 256 == 0) at the 256-row tile boundaries: a single row,
# one row short of / exactly / one past one and two pair tiles, with and
# without SiLU*up, LoRA ranks that leave a partial 64-wide LoRA stage.
PAIR_EDGES = [(M, 512, 512, rank, silu) for M in (1, 255, 256, 257, 511, 512, 513)
              for rank, silu in ((48, False), (80, True))]


@pytest.mark.parametrize("M,K,N,rank,silu", PAIR_EDGES)
def test_pair_tile_boundaries(M, K, N, rank, silu):
    p = synth.projection(3000 + M + rank, M, K, N, rank, outlier_frac=0.01)
    got, dev, pw = run(p, silu=silu)
    assert got.shape == (M, N // 2 if silu else N)
    assert_parity(got, ref(p, silu=silu), f"pair edge M={M} r={rank} silu={silu}")
    assert_bf16_is_rounded_f32(p, silu=silu, dev=dev, pw=pw)


def test_tiny_workload_matches_oracle():
    c = configs.TINY
    p = synth.projection(c["seed"], c["M"], c["K"], c["N"], c["rank"])
    got, _, _ = run(p)
    assert_parity(got, ref(p), "tiny")


@pytest.mark.parametrize("silu", [False, True])
def test_disabled_exactness_bitwise(silu):
    p = synth.projection(7, 333, 256, 512, 128)
    for dt in (torch.bfloat16, torch.float32):
        base, dev, pw = run(p, use_adapter=False, silu=silu, out_dtype=dt)
        zero, _, _ = run(p, strength=0.0, silu=silu, dev=dev, pw=pw, out_dtype=dt)
        assert np.array_equal(base.view(np.uint32), zero.view(np.uint32))
        one, _, _ = run(p, strength=1.0, silu=silu, dev=dev, pw=pw, out_dtype=dt)
        assert not np.array_equal(base, one)


def test_adapter_switching_per_call():
    M, K, N = 300, 256, 384
    p = synth.projection(11, M, K, N, 128)
    rng = np.random.default_rng(12)
    ad2 = synth.adapter(rng, N, K, 384)
    dev = to_dev(p)
    pw = h3lin.pack_weight(dev["W"])
    a1 = dev["adapter"]
    a2 = h3lin.Adapter(synth.to_bf16_tensor(ad2["A"]).cuda(), synth.to_bf16_tensor(ad2["B"]).cuda(), 384, 384.0)
    wref = linear.pack_weight(p["W"])
    outs = []
    for ad, s in [(a1, 1.0), (a2, 0.5), (None, 1.0), (a1, 1.0), (a2, 1.0)]:
        o = h3lin.forward(dev["x"], pw, dev["pqs"], ad, s, out_dtype=torch.float32)
        outs.append(o.cpu().numpy())
    for o, (ad, s) in zip(outs, [(p["adapter"], 1.0), (ad2, 0.5), (None, 1.0), (p["adapter"], 1.0), (ad2, 1.0)]):
        assert_parity(o, linear.forward(p["x"], wref, p["pqs"], ad, s), "switch")
    assert np.array_equal(outs[0], outs[3])        # no state carried between calls


def test_strength_linearity():
    p = synth.projection(21, 256, 256, 256, 64)
    y0, dev, pw = run(p, strength=0.0)
    yh, _, _ = run(p, strength=0.5, dev=dev, pw=pw)
    y1, _, _ = run(p, strength=1.0, dev=dev, pw=pw)
    assert_parity(yh, ref(p, 0.5), "s=0.5")
    d1, dh = y1.astype(np.float64) - y0, yh.astype(np.float64) - y0
    assert np.linalg.norm(d1 - 2 * dh) / np.linalg.norm(d1) < 1e-3


def test_zero_base_weight_is_pure_lora():
    p = synth.projection(31, 200, 256, 384, 32)
    p["W"] = np.zeros_like(p["W"])
    got, _, _ = run(p)
    assert_parity(got, ref(p), "pure LoRA")


def test_rows_beyond_M_untouched():
    p = synth.projection(41, 150, 256, 256, 16)
    dev = to_dev(p)
    pw = h3lin.pack_weight(dev["W"])
    for dt in (torch.bfloat16, torch.float32):
        big = torch.full((256, 256), 7.0, dtype=dt, device="cuda")
        h3lin.forward(dev["x"], pw, dev["pqs"], dev["adapter"], 1.0, False, out=big[:150])
        torch.cuda.synchronize()
        assert torch.all(big[150:] == 7.0)
        if dt == torch.float32:
            assert_parity(big[:150].cpu().numpy(), ref(p), "canary")


def test_device_status_clean():
    p = synth.projection(51, 100, 128, 128, 16)
    dev = to_dev(p)
    pw = h3lin.pack_weight(dev["W"])
    ws = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(100, 128, 128, 16))
    h3lin.forward(dev["x"], pw, dev["pqs"], dev["adapter"], 1.0, False, workspace=ws)
    assert h3lin.read_status(ws) == 0


def test_empty_input_is_a_no_op():
    """M = 0 rows: the forward and the quantiser accept it, enqueue nothing and
    return empty results; a following normal call is unaffected."""
    K, N, r = 256, 512, 16
    p = synth.projection(4242, 8, K, N, r)
    pw = h3lin.pack_weight(synth.to_bf16_tensor(p["W"]).cuda())
    a = p["adapter"]
    ad = h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), r, a["alpha"])
    s = torch.from_numpy(p["pqs"]).cuda()
    x0 = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    y0 = h3lin.forward(x0, pw, s, ad, 1.0)
    assert y0.shape == (0, N)
    y0s = h3lin.forward(x0, pw, s, ad, 1.0, silu_mul=True)
    assert y0s.shape == (0, N // 2)
    codes, scales, ts = h3lin.quantize_act(x0, s)
    assert codes.numel() == 0
    torch.cuda.synchronize()
    got, _, _ = run(p)
    assert_parity(got, ref(p), "after empty calls")
