"""Row counts where 32-bit element offsets overflow.

M = 3 500 037 rows of K = 5120 (x is 35.8 GB of bf16): a row's offset in
16-byte chunks, row * 640, passes 2^31 from row 3 355 444 on, so any index
product kept in 32 bits would land rows of the tail on the wrong data.  x
repeats a 256-row pattern (made on the device by torch from the pattern's
seeded values), so the oracle needs only the pattern: the tensor amax of the
whole x is the pattern's, every row is quantised like its pattern row, and
the projection of row r equals that of row r mod 256.  Checked on rows at
both ends and past the 2^31 boundary: tensor scale bit-exact, codes and
scale bytes bit-exact against the oracle, outputs bit-identical to the
pattern row's output and at the parity bar against the oracle."""
import numpy as np
import pytest

from tests._util import assert_parity, have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

torch = pytest.importorskip("torch")

from nvfp4_linear_lora_gb300 import build as h3build  # noqa: E402
from nvfp4_linear_lora_gb300 import h3lin, synth  # noqa: E402
from oracle import linear, nvfp4  # noqa: E402

M, K, N, RANK, P = 3_500_037, 5120, 256, 16, 256


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _rows():
    rng = np.random.default_rng(5)
    sample = rng.integers(3_355_444, M, 200)   # past the 2^31 chunk offset
    return np.unique(np.concatenate([np.arange(P), np.arange(M - P, M), sample]))


def _scale_offsets(rows, K):
    r = np.asarray(rows, np.int64)[:, None]
    j = np.arange(K // 16, dtype=np.int64)[None, :]
    rr = r % 128
    return ((r // 128) * (K // 64) + j // 4) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + j % 4


@pytest.fixture(scope="module")
def big():
    p = synth.projection(77, P, K, N, RANK, outlier_frac=0.01)
    xp = synth.to_bf16_tensor(p["x"]).cuda()
    x = xp.repeat((M + P - 1) // P, 1)[:M]
    assert x.is_contiguous() and x.shape == (M, K)
    a = p["adapter"]
    dev = dict(x=x, pqs=torch.from_numpy(p["pqs"]).cuda(), pw=h3lin.pack_weight(synth.to_bf16_tensor(p["W"]).cuda()),
               ad=h3lin.Adapter(synth.to_bf16_tensor(a["A"]).cuda(), synth.to_bf16_tensor(a["B"]).cuda(), a["rank"],
                                a["alpha"]))
    yield p, dev
    del dev
    torch.cuda.empty_cache()


def test_quantiser_past_32_bit_offsets(big):
    p, d = big
    codes, scales, ts = h3lin.quantize_act(d["x"], d["pqs"])
    torch.cuda.synchronize()
    rq, rs, rts = nvfp4.quantize(p["x"], p["pqs"])   # the pattern: same amax, same rows
    assert np.float32(ts.cpu().numpy()[0]) == rts
    rows = _rows()
    idx = torch.from_numpy(rows).cuda()
    got_codes = codes.index_select(0, idx).cpu().numpy()
    assert np.array_equal(got_codes, rq[rows % P])
    offs = torch.from_numpy(_scale_offsets(rows, K).reshape(-1)).cuda()
    got_sf = scales.index_select(0, offs).cpu().numpy().reshape(len(rows), K // 16)
    assert np.array_equal(got_sf, rs.reshape(P, K // 16)[rows % P])
    del codes, scales


def test_forward_past_32_bit_offsets(big):
    p, d = big
    out = h3lin.forward(d["x"], d["pw"], d["pqs"], d["ad"], 1.0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = _rows()
    got = out.index_select(0, torch.from_numpy(rows).cuda()).cpu().numpy()
    del out
    # every row equals its pattern row bit for bit (rows < P are the pattern)
    first = {r: i for i, r in enumerate(rows) if r < P}
    same = np.stack([got[first[r % P]] for r in rows])
    assert np.array_equal(got.view(np.uint32), same.view(np.uint32))
    ref = linear.forward(p["x"], linear.pack_weight(p["W"]), p["pqs"], p["adapter"], 1.0, False)
    assert_parity(got, ref[rows % P], "rows past 2^31 chunk offsets")
