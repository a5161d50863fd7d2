"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (one h3lin_forward per projection, full M, resident adapters).

The oracle evaluates full rows; at sizes where every row would take too long
it evaluates every row of the ragged last 128-row tile plus 512 seeded-random
rows, with the activation's tensor scale taken over the whole tensor.  The
quantised activation is checked bit-exactly on the same rows; outputs are
checked on the fp32 output mode against the parity bar."""
import numpy as np
import pytest

from tests._util import assert_parity, have_gpu, native_to_rowmajor

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import configs, h3lin, synth  # noqa: E402
from oracle import linear, nvfp4  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def sample_rows(M, seed, n_random=512):
    rng = np.random.default_rng(seed)
    tail0 = (M - 1) // 128 * 128
    rows = set(range(tail0, M)) | {0}
    rows |= set(rng.choice(M, min(n_random, M), replace=False).tolist())
    return np.array(sorted(rows))


class Proj:
    """One projection resident on the device plus its oracle-side weight."""

    def __init__(self, x, pqs, W, adapter, silu=False):
        self.x, self.pqs, self.W, self.adapter, self.silu = x, pqs, W, adapter, silu
        self.xd = synth.to_bf16_tensor(x).cuda()
        self.sd = torch.from_numpy(pqs).cuda() if pqs is not None else None
        self.pw = h3lin.pack_weight(synth.to_bf16_tensor(W).cuda())
        self.ad = None
        if adapter is not None:
            self.ad = h3lin.Adapter(synth.to_bf16_tensor(adapter["A"]).cuda(), synth.to_bf16_tensor(adapter["B"]).cuda(),
                                    adapter["rank"], adapter["alpha"])
        self.wref = linear.pack_weight(W)
        self.amax = nvfp4.tensor_amax_chunked(x, pqs)

    def gpu(self, rows, strength=1.0, adapter="own", out_dtype=torch.float32):
        ad = self.ad if adapter == "own" else adapter
        M = self.x.shape[0]
        ws = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(M, self.pw.K, self.pw.N, ad.rank if ad else 0))
        out = h3lin.forward(self.xd, self.pw, self.sd, ad, strength, self.silu, workspace=ws, out_dtype=out_dtype)
        torch.cuda.synchronize()
        assert h3lin.read_status(ws) == 0
        ts = np.float32(ws[4:8].cpu().numpy().view(np.float32)[0])
        idx = torch.from_numpy(rows).cuda()
        return out.index_select(0, idx).float().cpu().numpy(), ts, out

    def ref(self, rows, strength=1.0, adapter="own"):
        ad = self.adapter if adapter == "own" else adapter
        return linear.forward(self.x, self.wref, self.pqs, ad, strength, self.silu, rows=rows, x_amax=self.amax)

    def check_quant(self, rows):
        codes, scales, ts = h3lin.quantize_act(self.xd, self.sd)
        torch.cuda.synchronize()
        M, K = self.x.shape
        rq, rs, rts = nvfp4.quantize(self.x, self.pqs, rows=rows, amax=self.amax)
        assert np.float32(ts.cpu().numpy()[0]) == rts
        idx = torch.from_numpy(rows).cuda()
        np.testing.assert_array_equal(codes.index_select(0, idx).cpu().numpy(), rq)
        np.testing.assert_array_equal(native_to_rowmajor(scales.cpu().numpy(), M, K)[rows], rs)
        return rts


def test_qkv_9437_all_rows():
    c = configs.QKV
    p = synth.projection(c["seed"], c["M"], c["K"], c["N"], c["rank"], outlier_frac=c["outlier_frac"])
    pr = Proj(p["x"], p["pqs"], p["W"], p["adapter"])
    rows = np.arange(c["M"])
    rts = pr.check_quant(rows)
    got, ts, _ = pr.gpu(rows)
    assert ts == rts
    assert_parity(got, pr.ref(rows), "qkv 9437")


@pytest.fixture(scope="module")
def block():
    """The block's four projections at S = 37726 (down gets its own N(0,1) input)."""
    S = configs.BLOCK_S
    rng = np.random.default_rng(configs.BLOCK_SEED)
    out = {}
    for name, K, N, r, silu in configs.BLOCK_PROJECTIONS:
        x = synth.activation(rng, S, K)
        s = synth.pre_quant_scale(rng, K)
        W = synth.weight(rng, N, K)
        ad = synth.adapter(rng, N, K, r)
        out[name] = Proj(x, s, W, ad, silu)
    return out


@pytest.mark.parametrize("name", [p[0] for p in configs.BLOCK_PROJECTIONS])
def test_block_projection_S37726(block, name):
    pr = block[name]
    rows = sample_rows(configs.BLOCK_S, 100 + len(name))
    rts = pr.check_quant(rows)
    got, ts, full = pr.gpu(rows)
    assert ts == rts
    assert_parity(got, pr.ref(rows), f"block {name}")
    # the bf16 output the benchmark stores is the rounding of this fp32 output
    b16, _, _ = pr.gpu(rows, out_dtype=torch.bfloat16)
    assert np.array_equal(b16, torch.from_numpy(got).to(torch.bfloat16).float().numpy())


def test_block_chain_deterministic(block):
    """Back-to-back block runs (bench launch configuration, bf16 outputs,
    down consuming gate/up's output) reproduce bit-identical outputs."""
    gu, dn = block["gate_up"], block["down"]
    outs = []
    for _ in range(2):
        h = h3lin.forward(gu.xd, gu.pw, gu.sd, gu.ad, 1.0, True)
        y = h3lin.forward(h, dn.pw, dn.sd, dn.ad, 1.0, False)
        torch.cuda.synchronize()
        outs.append((h.view(torch.int16).clone(), y.view(torch.int16).clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.fixture(scope="module")
def switching():
    c = configs.QKV
    S = configs.SWITCH_S
    p = synth.projection(configs.SWITCH_SEED, S, c["K"], c["N"], c["rank"], outlier_frac=c["outlier_frac"],
                         with_adapter=False)
    ads = [synth.adapter(np.random.default_rng(sd), c["N"], c["K"], r)
           for sd, r in zip(configs.SWITCH_ADAPTER_SEEDS, (384, 128))]
    pr = Proj(p["x"], p["pqs"], p["W"], None)
    dev_ads = [h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), a["rank"],
                             a["alpha"]) for a in ads]
    return pr, ads, dev_ads


def test_switch_disabled_exactness_bitwise(switching):
    pr, ads, dev_ads = switching
    rows = np.arange(4)
    _, _, base = pr.gpu(rows, adapter=None, out_dtype=torch.bfloat16)
    base = base.view(torch.int16).clone()
    for a in dev_ads:
        _, _, z = pr.gpu(rows, strength=0.0, adapter=a, out_dtype=torch.bfloat16)
        assert torch.equal(z.view(torch.int16), base)


@pytest.mark.parametrize("which,strength", [(0, 0.5), (0, 1.0), (1, 0.5), (1, 1.0), (None, 1.0)])
def test_switch_adapters_per_call(switching, which, strength):
    pr, ads, dev_ads = switching
    rows = sample_rows(configs.SWITCH_S, 200 + (which or 0))
    # interleave a call with the other adapter first: nothing may carry over
    other = dev_ads[1 - which] if which is not None else dev_ads[0]
    pr.gpu(rows[:2], 1.0, adapter=other)
    got, _, _ = pr.gpu(rows, strength, adapter=dev_ads[which] if which is not None else None)
    want = pr.ref(rows, strength, adapter=ads[which] if which is not None else None)
    assert_parity(got, want, f"switch adapter={which} strength={strength}")


@pytest.mark.parametrize("i", range(len(configs.SWEEP_M)))
def test_sequence_sweep_student_t(i):
    M, seed = configs.SWEEP_M[i], configs.SWEEP_SEEDS[i]
    c = configs.QKV
    p = synth.projection(seed, M, c["K"], c["N"], c["rank"], law="student_t3", outlier_frac=0.01)
    pr = Proj(p["x"], p["pqs"], p["W"], p["adapter"])
    rows = np.arange(M) if M <= 4096 else sample_rows(M, 300 + i)
    rts = pr.check_quant(rows)
    got, ts, _ = pr.gpu(rows)
    assert ts == rts
    assert_parity(got, pr.ref(rows), f"sweep M={M}")
