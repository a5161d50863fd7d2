"""Failure detection on the GPU without a fault: a bounded device wait that
nothing satisfies expires, the kernel records H3LIN_E_TIMEOUT in the
workspace status word and returns; the host reads it, clears it, and the
same context then runs a normal projection correctly."""
import numpy as np
import pytest

from tests._util import assert_parity, have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import h3lin, synth  # noqa: E402
from oracle import linear  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def test_device_wait_timeout_is_reported_and_context_survives():
    stream = torch.cuda.current_stream().cuda_stream
    ws = h3lin.new_workspace(h3lin.h3lin_quant_workspace_bytes())
    assert h3lin.read_status(ws) == h3lin.H3LIN_OK
    st = h3lin.h3lin_selftest_wait_timeout(ws.data_ptr(), ws.numel(), 1 << 22, stream)   # ~2 ms
    assert st == h3lin.H3LIN_OK
    assert h3lin.read_status(ws) == h3lin.H3LIN_E_TIMEOUT
    # sticky until cleared
    assert h3lin.read_status(ws) == h3lin.H3LIN_E_TIMEOUT
    assert h3lin.h3lin_workspace_init(ws.data_ptr(), ws.numel(), stream) == h3lin.H3LIN_OK
    assert h3lin.read_status(ws) == h3lin.H3LIN_OK

    # the context is healthy: a normal projection still matches the oracle
    p = synth.projection(77, 300, 256, 512, 32)
    x = synth.to_bf16_tensor(p["x"]).cuda()
    s = torch.from_numpy(p["pqs"]).cuda()
    pw = h3lin.pack_weight(synth.to_bf16_tensor(p["W"]).cuda())
    a = p["adapter"]
    ad = h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), a["rank"], a["alpha"])
    fws = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(300, 256, 512, 32))
    y = h3lin.forward(x, pw, s, ad, 1.0, out_dtype=torch.float32, workspace=fws)
    assert h3lin.read_status(fws) == h3lin.H3LIN_OK
    ref = linear.forward(p["x"], linear.pack_weight(p["W"]), p["pqs"], a, 1.0)
    assert_parity(y.cpu().numpy(), ref, "after timeout")


def test_selftest_rejects_bad_arguments():
    stream = torch.cuda.current_stream().cuda_stream
    ws = h3lin.new_workspace(h3lin.h3lin_quant_workspace_bytes())
    assert h3lin.h3lin_selftest_wait_timeout(None, 0, 1000, stream) == h3lin.H3LIN_E_INVALID
    assert h3lin.h3lin_selftest_wait_timeout(ws.data_ptr(), 16, 1000, stream) == h3lin.H3LIN_E_WORKSPACE
    assert h3lin.h3lin_selftest_wait_timeout(ws.data_ptr(), ws.numel(), 0, stream) == h3lin.H3LIN_E_INVALID
    assert h3lin.read_status(ws) == h3lin.H3LIN_OK
