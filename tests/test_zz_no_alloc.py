"""The allocation-free forward entry point (h3lin_forward_noalloc), for
callers that cannot call cudaMalloc (a plugin whose host application owns all
device memory, a loop where allocation is forbidden).  Its scratch is a fixed
array inside the library that every call shares, so each call must give
exactly the bytes h3lin_forward gives with a fresh caller-provided workspace,
whatever the previous call left in the array: consecutive calls here change
M (down as well as up), the rank, the epilogue and adapter/NULL.  The
scratch's status word must read OK afterwards, and work larger than the
scratch is refused.

Collected last on purpose: it runs after every other test file, and also
passes when run alone in a fresh process."""
import pytest

from tests._util import have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import h3lin, synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _setup(seed, M, K, N, rank):
    p = synth.projection(seed, M, K, N, rank, outlier_frac=0.01)
    x = synth.to_bf16_tensor(p["x"]).cuda()
    s = torch.from_numpy(p["pqs"]).cuda()
    pw = h3lin.pack_weight(synth.to_bf16_tensor(p["W"]).cuda())
    a = p["adapter"]
    ad = h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), a["rank"], a["alpha"])
    return x, s, pw, ad


def _noalloc(x, s, pw, ad, silu, out, dtype):
    st = h3lin.h3lin_forward_noalloc(x.data_ptr(), x.shape[0], s.data_ptr(), pw.c_struct(),
                                     h3lin.H3LIN_EPI_SILU_MUL if silu else h3lin.H3LIN_EPI_NONE,
                                     ad.c_struct() if ad is not None else None, 1.0, out.data_ptr(),
                                     h3lin.H3LIN_OUT_F32 if dtype == torch.float32 else h3lin.H3LIN_OUT_BF16,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == h3lin.H3LIN_OK, h3lin.h3lin_status_string(st)


# (M, K, N, rank, SiLU*up, adapter on, output dtype): M rises and falls, the
# rank and the epilogue change, a base-only call sits between adapter calls
SEQUENCE = [
    (1000, 1024, 1280, 128, False, True, torch.float32),
    (515, 512, 512, 384, True, True, torch.float32),
    (1000, 1024, 1280, 128, False, False, torch.float32),
    (2048, 1024, 1280, 128, False, True, torch.bfloat16),
    (300, 1024, 1280, 128, False, True, torch.float32),
    (515, 512, 512, 384, True, False, torch.bfloat16),
]


def test_noalloc_bit_identical_to_workspace_forward_on_consecutive_calls():
    cache = {}
    for M, K, N, rank, silu, on, dtype in SEQUENCE:
        key = (M, K, N, rank)
        if key not in cache:
            cache[key] = _setup(M + N + rank, M, K, N, rank)
        x, s, pw, ad = cache[key]
        ad = ad if on else None
        want = h3lin.forward(x, pw, s, ad, 1.0, silu, out_dtype=dtype)
        n_out = N // 2 if silu else N
        for _ in range(2):   # two calls in a row on the same shared scratch
            got = torch.full((M, n_out), float("nan"), dtype=dtype, device="cuda")
            _noalloc(x, s, pw, ad, silu, got, dtype)
            torch.cuda.synchronize()
            assert torch.equal(got, want), f"noalloc differs from h3lin_forward at M={M} N={N} rank={rank} " \
                                           f"silu={silu} adapter={on} {dtype}"
    st, word = h3lin.h3lin_noalloc_read_status(torch.cuda.current_stream().cuda_stream)
    assert st == h3lin.H3LIN_OK and word == h3lin.H3LIN_OK, (st, word)


def test_noalloc_rejects_work_beyond_its_scratch():
    K, N = 5120, 15360
    M = 1 + h3lin.H3LIN_NOALLOC_SCRATCH_BYTES // (K // 2)          # codes alone exceed the scratch
    assert h3lin.h3lin_forward_workspace_bytes(M, K, N, 0) > h3lin.H3LIN_NOALLOC_SCRATCH_BYTES
    w = h3lin.h3lin_weight(0x10000, 0x10000, 0x10000, N, K)
    st = h3lin.h3lin_forward_noalloc(0x10000, M, None, w, 0, None, 1.0, 0x10000, 0,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == h3lin.H3LIN_E_WORKSPACE
