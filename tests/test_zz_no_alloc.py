"""The allocation-free forward entry point (h3lin_forward_noalloc), for
callers that cannot call cudaMalloc: it must give the same output as
h3lin_forward with a caller-provided workspace, on consecutive calls that
share its fixed in-library scratch, and refuse work larger than that scratch.

Collected last on purpose: it runs after every other test file, and also
passes when run alone in a fresh process."""
import numpy as np
import pytest

from tests._util import assert_parity, have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import h3lin, synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _setup(seed, M, K, N, rank, silu):
    p = synth.projection(seed, M, K, N, rank, outlier_frac=0.01)
    x = synth.to_bf16_tensor(p["x"]).cuda()
    s = torch.from_numpy(p["pqs"]).cuda()
    pw = h3lin.pack_weight(synth.to_bf16_tensor(p["W"]).cuda())
    a = p["adapter"]
    ad = h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), a["rank"], a["alpha"])
    return x, s, pw, ad


def _noalloc(x, s, pw, ad, silu, out):
    st = h3lin.h3lin_forward_noalloc(x.data_ptr(), x.shape[0], s.data_ptr(), pw.c_struct(),
                                     h3lin.H3LIN_EPI_SILU_MUL if silu else h3lin.H3LIN_EPI_NONE,
                                     ad.c_struct() if ad is not None else None, 1.0, out.data_ptr(),
                                     h3lin.H3LIN_OUT_F32, torch.cuda.current_stream().cuda_stream)
    assert st == h3lin.H3LIN_OK, h3lin.h3lin_status_string(st)


@pytest.mark.parametrize("M,K,N,rank,silu", [(1000, 1024, 1280, 128, False), (515, 512, 512, 384, True)])
def test_noalloc_matches_workspace_forward_twice(M, K, N, rank, silu):
    x, s, pw, ad = _setup(M + N, M, K, N, rank, silu)
    want = h3lin.forward(x, pw, s, ad, 1.0, silu, out_dtype=torch.float32)
    n_out = N // 2 if silu else N
    for _ in range(2):   # consecutive calls share the scratch
        got = torch.full((M, n_out), float("nan"), dtype=torch.float32, device="cuda")
        _noalloc(x, s, pw, ad, silu, got)
        torch.cuda.synchronize()
        assert_parity(got.cpu().numpy(), want.cpu().numpy(), "noalloc vs workspace forward")
    # a base-only call in between, then the adapter call again
    base = torch.empty((M, n_out), dtype=torch.float32, device="cuda")
    _noalloc(x, s, pw, None, silu, base)
    again = torch.empty((M, n_out), dtype=torch.float32, device="cuda")
    _noalloc(x, s, pw, ad, silu, again)
    torch.cuda.synchronize()
    assert_parity(again.cpu().numpy(), want.cpu().numpy(), "noalloc after base call")
    assert_parity(base.cpu().numpy(), h3lin.forward(x, pw, s, None, 1.0, silu, out_dtype=torch.float32).cpu().numpy(),
                  "noalloc base")


def test_noalloc_rejects_work_beyond_its_scratch():
    K, N = 5120, 15360
    M = 1 + h3lin.H3LIN_NOALLOC_SCRATCH_BYTES // (K // 2)          # codes alone exceed the scratch
    assert h3lin.h3lin_forward_workspace_bytes(M, K, N, 0) > h3lin.H3LIN_NOALLOC_SCRATCH_BYTES
    w = h3lin.h3lin_weight(0x10000, 0x10000, 0x10000, N, K)
    st = h3lin.h3lin_forward_noalloc(0x10000, M, None, w, 0, None, 1.0, 0x10000, 0,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == h3lin.H3LIN_E_WORKSPACE
