"""GPU parity of the quantiser: codes, scales and tensor scale bit-exact
against the oracle (through the C ABI)."""
import numpy as np
import pytest

from tests._util import have_gpu, native_to_rowmajor

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import h3lin, synth  # noqa: E402
from oracle import nvfp4  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def gpu_quantize(x, s):
    M, K = x.shape
    xt = synth.to_bf16_tensor(x).cuda()
    st = torch.from_numpy(s).cuda() if s is not None else None
    codes, scales, ts = h3lin.quantize_act(xt, st)
    torch.cuda.synchronize()
    raw = scales.cpu().numpy()
    return codes.cpu().numpy(), native_to_rowmajor(raw, M, K), np.float32(ts.cpu().numpy()[0]), raw


def check_exact(x, s):
    M, K = x.shape
    c, sc, ts, raw = gpu_quantize(x, s)
    rc, rsc, rts = nvfp4.quantize(x, s)
    assert ts == rts, (ts, rts)
    np.testing.assert_array_equal(sc, rsc)
    np.testing.assert_array_equal(c, rc)
    # padded rows of the last 128-row atom hold scale 0
    mpad = (M + 127) // 128 * 128
    if mpad > M:
        from tests._util import native_scale_offsets
        pad = native_scale_offsets(mpad, K)[M:]
        assert not raw[pad].any()


@pytest.mark.parametrize("M,K", [(1, 64), (37, 64), (127, 128), (128, 256), (129, 192), (200, 256),
                                 (300, 1024), (1000, 5120), (2053, 320)])
@pytest.mark.parametrize("with_pqs", [True, False])
def test_quantize_bit_exact(M, K, with_pqs):
    rng = np.random.default_rng(M * 7 + K)
    x = synth.activation(rng, M, K, "normal", 0.01)
    s = synth.pre_quant_scale(rng, K) if with_pqs else None
    check_exact(x, s)


def test_quantize_student_t_outliers():
    rng = np.random.default_rng(3)
    x = synth.activation(rng, 517, 5120, "student_t3", 0.01)
    check_exact(x, synth.pre_quant_scale(rng, 5120))


def test_quantize_special_values():
    rng = np.random.default_rng(9)
    M, K = 260, 256
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[3] = 0.0                                   # zero row
    x[5, :16] = 1e-30                            # block far below the tensor scale
    x[6, 16:32] = -1e-6                          # tiny negatives -> code 0x8 or small
    x[7, 32:48] = 5.0                            # identical values
    x[8, 0] = 3.0e4                              # outlier: sets the tensor amax
    x[9, 48:64] = -0.0
    check_exact(synth.bf16_round(x), None)


def test_quantize_exact_ties():
    """Blocks with power-of-two scales whose elements sit exactly on E2M1 ties."""
    M, K = 130, 128
    ts = 2.0 ** -4
    ties = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, 0.5])
    x = np.zeros((M, K))
    for r in range(M):
        for b in range(K // 16):
            k = 2.0 ** ((r + b) % 7 - 3)
            x[r, 16 * b:16 * b + 16] = np.roll(ties, r % 16) * k * ts
    x[0, 0] = 2688.0 * ts
    x = x.astype(np.float32)
    assert np.array_equal(synth.bf16_round(x), x)
    check_exact(x, None)


def test_quantize_all_zero_tensor():
    x = np.zeros((64, 128), np.float32)
    c, sc, ts, _ = gpu_quantize(x, None)
    assert ts == 1.0 and not c.any() and not sc.any()


@pytest.mark.parametrize("N,K", [(384, 256), (256, 5120), (15360, 5120)])
def test_pack_weight_bit_exact(N, K):
    rng = np.random.default_rng(N + K)
    W = synth.weight(rng, N, K)
    pw = h3lin.pack_weight(synth.to_bf16_tensor(W).cuda())
    torch.cuda.synchronize()
    rc, rsc, rts = nvfp4.quantize(W, None)
    assert np.float32(pw.tensor_scale.cpu().numpy()[0]) == rts
    np.testing.assert_array_equal(pw.codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(native_to_rowmajor(pw.scales.cpu().numpy(), N, K), rsc)
