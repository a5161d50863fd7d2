"""The bounds-checked build (libh3lin_bounds.so, compiled with -DH3LIN_BOUNDS)
on the GPU: its index checks are live (the self-test's out-of-range store is
reported as H3LIN_E_BOUNDS and skipped), and the hot-path parity tests pass
with it loaded, with no index ever leaving its buffer (every workspace's
status word stays 0) and every guard tail intact.  compute-sanitizer is
closed on this pool; these checks and the canaries stand in for it."""
import os
import subprocess
import sys

import pytest

from tests._util import have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(code_or_args, pytest_run=False):
    env = dict(os.environ, H3LIN_BOUNDS="1", H3LIN_CANARY="1")
    if pytest_run:
        cmd = [sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu"] + code_or_args
    else:
        cmd = [sys.executable, "-c", code_or_args]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)


@pytest.fixture(scope="module", autouse=True)
def built():
    from nvfp4_linear_lora_gb300 import build as h3build
    h3build.build(bounds=True)


def test_bounds_check_is_live():
    code = """
import torch
from nvfp4_linear_lora_gb300 import h3lin
assert h3lin.h3lin_bounds_build() == 1
ws = h3lin.new_workspace(h3lin.h3lin_quant_workspace_bytes())
before = ws[512:2048].clone()
st = h3lin.h3lin_selftest_bounds(ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
assert st == h3lin.H3LIN_OK, st
assert h3lin.read_status(ws) == h3lin.H3LIN_E_BOUNDS
assert torch.equal(ws[512:2048], before), "the out-of-range store was not skipped"
h3lin._bounds_ws.clear()   # this workspace holds the error on purpose
print("bounds self-test ok")
"""
    r = _run(code)
    assert r.returncode == 0 and "bounds self-test ok" in r.stdout, r.stdout + r.stderr


def test_hot_path_parity_under_the_bounds_build():
    # the projection, quantiser, MLP fusion, LoRA isolation and the steps
    # around the block, with every plain global index checked
    files = ["tests/test_gpu_quant.py", "tests/test_gpu_forward.py", "tests/test_gpu_mlp.py",
             "tests/test_gpu_modulate.py", "tests/test_gpu_rope.py", "tests/test_gpu_lora.py",
             "-k", "not S37726 and not full_size and not block"]
    r = _run(files, pytest_run=True)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_launch_trace_lists_every_kernel_of_a_forward():
    code = """
import torch
from nvfp4_linear_lora_gb300 import h3lin
x = torch.randn(300, 512, device="cuda").to(torch.bfloat16)
w = (torch.randn(512, 512, device="cuda") / 23).to(torch.bfloat16)
A = (torch.randn(64, 512, device="cuda") / 23).to(torch.bfloat16)
B = (torch.randn(512, 64, device="cuda") / 80).to(torch.bfloat16)
pw = h3lin.pack_weight(w)
h3lin.forward(x, pw, None, h3lin.Adapter(A, B, 64, 64.0), 1.0)
torch.cuda.synchronize()
"""
    env = dict(os.environ, H3LIN_TRACE="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("h3lin: ")]
    names = [ln.split()[1] for ln in lines]
    # packing: amax + quantise; forward: amax with A(x), quantise, the CTA-pair GEMM
    assert names == ["k_amax", "k_quant", "k_amax_lora<amax>", "k_quant", "k_fp4gemm_pair"], names
    gemm = lines[-1]
    for field in ("grid=", "cluster=2", "block=", "smem=", "M=300", "N=512", "K=512", "rank=64", "raster_group="):
        assert field in gemm, gemm
