"""Modulation producer on the GPU against the oracle, and the produced
projection against the unfused one.

x_mod: fp32 LayerNorm and modulation then one bf16 rounding on the GPU, float64
then one rounding in the oracle: per element one bf16 unit (2^-8 of the
value covers the rounding and the fp32 work before it) plus 2e-4 absolute
for the fp32 row statistics over K <= 8192 values.  The projection that reads
the producer's amax partials must be bit-identical to h3lin_forward on the
same x_mod (max is exact; the codes, scales and tensor scale follow)."""
import numpy as np
import pytest

from tests._util import have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import configs, h3lin, synth  # noqa: E402
from oracle import modulation  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _inputs(seed, M, K, sizes):
    rng = np.random.default_rng(seed)
    x = synth.residual(rng, M, K)
    table = synth.adaln_table(rng, len(sizes), K)
    rows = synth.segment_rows(sizes)
    return x, table, rows, rng


def _check_xmod(got, x, table, rows, eps):
    ref = modulation.modulate(x, table, rows, eps, round_bf16=False)
    diff = np.abs(np.asarray(got, np.float64) - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2e-4 * (1.0 + np.abs(ref))
    assert np.all(diff <= bound), f"worst excess {(diff - bound).max():.3e}"
    # most elements land on the oracle's own bf16 rounding
    exact = np.mean(np.asarray(got, np.float32) == modulation.modulate(x, table, rows, eps))
    assert exact >= 0.99, f"exact fraction {exact:.4f}"


def _modulate(x, table, rows, ws, pqs=None, eps=1e-6):
    xd = synth.to_bf16_tensor(x).cuda()
    return h3lin.modulate_produce(xd, torch.from_numpy(table).cuda(), torch.from_numpy(rows).cuda(), ws,
                                  None if pqs is None else torch.from_numpy(pqs).cuda(), eps)


@pytest.mark.parametrize("M,K,sizes,eps", [(300, 1024, (200, 60, 40), 1e-6), (1, 64, (1,), 1e-6),
                                           (129, 8192, (100, 29), 1e-5), (1000, 5120, (1000,), 0.0)])
def test_modulate_matches_oracle(M, K, sizes, eps):
    x, table, rows, _ = _inputs(M + K, M, K, sizes)
    ws = h3lin.new_workspace(h3lin.h3lin_quant_workspace_bytes())
    got = _modulate(x, table, rows, ws, eps=eps)
    torch.cuda.synchronize()
    assert h3lin.read_status(ws) == 0
    _check_xmod(got.float().cpu().numpy(), x, table, rows, eps)


@pytest.mark.parametrize("with_adapter,with_pqs,f32", [(True, True, False), (False, True, True), (True, False, True)])
def test_produced_projection_is_bitwise_the_unfused_one(with_adapter, with_pqs, f32):
    M, K, N, r = 517, 1024, 1536, 64
    x, table, rows, rng = _inputs(7, M, K, (300, 200, 17))
    s = synth.pre_quant_scale(rng, K) if with_pqs else None
    W = synth.weight(rng, N, K)
    a = synth.adapter(rng, N, K, r)
    pw = h3lin.pack_weight(synth.to_bf16_tensor(W).cuda())
    ad = h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), r,
                       a["alpha"]) if with_adapter else None
    sd = torch.from_numpy(s).cuda() if with_pqs else None
    ws = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(M, K, N, r))
    xm = _modulate(x, table, rows, ws, s)
    dt = torch.float32 if f32 else torch.bfloat16
    y_prod = h3lin.forward_produced(xm, pw, ws, sd, ad, out_dtype=dt)
    torch.cuda.synchronize()
    assert h3lin.read_status(ws) == 0
    ts_prod = np.float32(ws[4:8].cpu().numpy().view(np.float32)[0])
    y_ref = h3lin.forward(xm, pw, sd, ad, out_dtype=dt)
    torch.cuda.synchronize()
    view = torch.int32 if f32 else torch.int16
    assert torch.equal(y_prod.view(view), y_ref.view(view))
    # the tensor scale from the producer's partials is the rule's, amax|x_mod * s| / 2688,
    # on the x_mod it produced (a property of the GPU's own output; no oracle input)
    prod = xm.float() * (sd if sd is not None else 1.0)
    amax = np.float32(prod.abs().max().item())
    want = np.float32(amax / np.float32(2688.0))
    want = want if want != 0 else np.float32(1.0)
    assert ts_prod == want


def test_bad_table_index_is_recorded_and_zeroed():
    M, K = 40, 256
    x, table, rows, _ = _inputs(11, M, K, (40,))
    rows = rows.copy()
    rows[5] = 3          # table has 1 row
    rows[17] = -1
    ws = h3lin.new_workspace(h3lin.h3lin_quant_workspace_bytes())
    got = _modulate(x, table, rows, ws).float().cpu().numpy()
    assert h3lin.read_status(ws) == h3lin.H3LIN_E_INVALID
    assert np.all(got[[5, 17]] == 0)
    keep = np.setdiff1d(np.arange(M), [5, 17])
    _check_xmod(got[keep], x[keep], table, rows[keep], 1e-6)
    h3lin.h3lin_workspace_init(ws.data_ptr(), ws.numel(), h3lin._stream())
    assert h3lin.read_status(ws) == 0


def test_empty_is_a_no_op():
    ws = h3lin.new_workspace(h3lin.h3lin_quant_workspace_bytes())
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    t = torch.zeros((1, 2, 256), dtype=torch.float32, device="cuda")
    r = torch.zeros((0,), dtype=torch.int32, device="cuda")
    h3lin.modulate_produce(x, t, r, ws)
    torch.cuda.synchronize()
    assert h3lin.read_status(ws) == 0


def test_block_S37726_segments_and_produced_qkv():
    """The block's QKV input at full size: three segments, sampled rows of
    x_mod against the oracle, the produced QKV projection bit-identical."""
    S, K = configs.BLOCK_S, configs.HIDDEN
    c = configs.MODULATION
    x, table, rows, rng = _inputs(configs.MODULATION_SEED, S, K, c["segments"])
    s = synth.pre_quant_scale(rng, K)
    N, r = 3 * K, 384
    W = synth.weight(rng, N, K)
    a = synth.adapter(rng, N, K, r)
    pw = h3lin.pack_weight(synth.to_bf16_tensor(W).cuda())
    ad = h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), r, a["alpha"])
    sd = torch.from_numpy(s).cuda()
    ws = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(S, K, N, r))
    xm = _modulate(x, table, rows, ws, s, c["eps"])
    y_prod = h3lin.forward_produced(xm, pw, ws, sd, ad)
    torch.cuda.synchronize()
    assert h3lin.read_status(ws) == 0
    samp = np.array(sorted(set(np.random.default_rng(4).choice(S, 512, replace=False).tolist())
                           | {0, S - 1} | set(np.cumsum(c["segments"])[:-1].tolist())))
    _check_xmod(xm.index_select(0, torch.from_numpy(samp).cuda()).float().cpu().numpy(), x[samp], table, rows[samp],
                c["eps"])
    y_ref = h3lin.forward(xm, pw, sd, ad)
    torch.cuda.synchronize()
    assert torch.equal(y_prod.view(torch.int16), y_ref.view(torch.int16))
