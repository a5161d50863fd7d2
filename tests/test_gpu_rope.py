"""Q/K RMSNorm + split-half three-axis RoPE on the GPU against the oracle.

The kernel computes in fp32 and stores bf16, the oracle in float64, so the
bound per element is one bf16 rounding (2^-9 of the value, taken as 2^-8 to
cover the fp32 rounding before it) plus the angle error carried by the pair:
angles are float(pos) * float(freq) in fp32, off by up to |angle| * 2^-23,
which moves each output by at most that times the pair's magnitude, plus a
few fp32 roundings of the normalised values (1e-5 of the pair).  V and the
rows past M must come back bit for bit."""
import numpy as np
import pytest

from tests._util import have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import configs, h3lin, synth  # noqa: E402
from oracle import rope  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _check(got, ref, qkv_in, pos, heads, rot, axis_dims, theta):
    """Element bound on Q and K, exact V."""
    HD = heads * 128
    got = np.asarray(got, np.float64)
    assert np.array_equal(got[:, 2 * HD:], qkv_in[:, 2 * HD:]), "V changed"
    h = rot // 2
    max_ang = float(np.max(np.abs(rope.angles(pos, axis_dims, theta)))) if len(pos) else 0.0
    ang_tol = max_ang * 2.0 ** -22 + 1e-6
    for part in (0, 1):
        g = got[:, part * HD:(part + 1) * HD].reshape(len(got), heads, 128)
        r = ref[:, part * HD:(part + 1) * HD].reshape(len(got), heads, 128)
        pair = np.abs(r).copy()
        mag = np.sqrt(r[..., :h] ** 2 + r[..., h:rot] ** 2)
        pair[..., :h] = mag
        pair[..., h:rot] = mag
        bound = 2.0 ** -8 * np.abs(r) + (ang_tol + 1e-5) * pair + 1e-30
        excess = np.abs(g - r) - bound
        assert np.all(excess <= 0), f"part {part}: worst excess {excess.max():.3e}"


def _run(M, heads, rot, axis_dims, theta, eps, seed, pos=None, pad_rows=3):
    rng = np.random.default_rng(seed)
    HD = heads * 128
    qkv = synth.activation(rng, M + pad_rows, 3 * HD)              # bf16 values
    wq, wk = synth.norm_gain(rng, 128), synth.norm_gain(rng, 128)
    if pos is None:
        pos = synth.rope_positions(M, frames=3, height=5, width=7)
    dev = synth.to_bf16_tensor(qkv).cuda()
    h3lin.qk_norm_rope(dev[:M] if M else dev[:0], torch.from_numpy(wq).cuda(), torch.from_numpy(wk).cuda(),
                       torch.from_numpy(np.ascontiguousarray(pos, np.int32)).cuda(), heads, rot, axis_dims, theta, eps)
    torch.cuda.synchronize()
    out = dev.float().cpu().numpy()
    assert np.array_equal(out[M:], qkv[M:]), "rows past M changed"
    ref = rope.qk_norm_rope(qkv[:M], heads, wq, wk, pos, 128, rot, axis_dims, theta, eps)
    _check(out[:M], ref, qkv[:M], pos, heads, rot, axis_dims, theta)


@pytest.mark.parametrize("M,heads,rot,axis_dims,theta,eps", [
    (300, 40, 96, (32, 32, 32), 10000.0, 1e-6),
    (1, 3, 96, (32, 32, 32), 10000.0, 1e-6),
    (37, 2, 128, (64, 32, 32), 500.0, 1e-5),
    (129, 5, 16, (0, 16, 0), 10000.0, 0.0),
    (64, 1, 48, (16, 0, 32), 10000.0, 1e-6),
])
def test_qk_norm_rope_matches_oracle(M, heads, rot, axis_dims, theta, eps):
    _run(M, heads, rot, axis_dims, theta, eps, seed=M + heads + rot)


def test_empty_is_a_no_op():
    _run(0, 4, 96, (32, 32, 32), 10000.0, 1e-6, seed=1, pos=np.zeros((0, 3), np.int32))


def test_large_positions():
    """Angles up to ~1e4 rad: the fp32 angle error stays inside the bound."""
    M = 64
    pos = np.stack([np.arange(M) * 150, np.arange(M) * 7, np.arange(M) % 11], axis=1).astype(np.int32)
    _run(M, 8, 96, (32, 32, 32), 10000.0, 1e-6, seed=9, pos=pos)


def test_block_S37726_sampled_rows():
    """The block's QKV output size and positions (40 heads, 96 rotated dims)."""
    c = configs.ROPE
    S = configs.BLOCK_S
    rng = np.random.default_rng(configs.ROPE_SEED)
    HD = c["heads"] * 128
    qkv = synth.activation(rng, S, 3 * HD)
    wq, wk = synth.norm_gain(rng, 128), synth.norm_gain(rng, 128)
    pos = synth.rope_positions(S, c["frames"], c["height"], c["width"])
    dev = synth.to_bf16_tensor(qkv).cuda()
    h3lin.qk_norm_rope(dev, torch.from_numpy(wq).cuda(), torch.from_numpy(wk).cuda(), torch.from_numpy(pos).cuda(),
                       c["heads"], c["rot"], c["axis_dims"], c["theta"], c["eps"])
    torch.cuda.synchronize()
    rows = np.array(sorted(set(np.random.default_rng(3).choice(S, 512, replace=False).tolist())
                           | set(range(S - 130, S)) | {0}))
    got = dev.index_select(0, torch.from_numpy(rows).cuda()).float().cpu().numpy()
    ref = rope.qk_norm_rope(qkv[rows], c["heads"], wq, wk, pos[rows], 128, c["rot"], c["axis_dims"], c["theta"],
                            c["eps"])
    _check(got, ref, qkv[rows], pos[rows], c["heads"], c["rot"], c["axis_dims"], c["theta"])
