"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point declared in include/h3lin.h, sizes are right, and invalid
arguments are rejected on the host before anything is enqueued."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from nvfp4_linear_lora_gb300 import build as h3build
from nvfp4_linear_lora_gb300 import h3lin

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    h3build.build()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "h3lin.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(h3lin_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ["h3lin_pack_weight", "h3lin_quantize_act", "h3lin_forward", "h3lin_read_status"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    L = h3lin.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_abi_version_and_strings():
    assert h3lin.h3lin_abi_version() == 1
    for s in range(8):
        assert len(h3lin.h3lin_status_string(s)) > 0


def test_sizes():
    assert h3lin.h3lin_codes_bytes(200, 256) == 200 * 128
    assert h3lin.h3lin_scales_bytes(200, 256) == 256 * 16
    assert h3lin.h3lin_scales_bytes(37726, 5120) == 37760 * 320
    assert h3lin.h3lin_codes_bytes(10, 100) == 0 and h3lin.h3lin_scales_bytes(0, 64) == 0
    ws = h3lin.h3lin_forward_workspace_bytes(9437, 5120, 15360, 384)
    need = 9437 * 2560 + 9472 * 320 + 9437 * 384 * 2 + 15360 * 384 * 2
    assert need < ws < need + 64 * 1024
    assert h3lin.h3lin_forward_workspace_bytes(9437, 5120, 15360, 0) < ws


def test_workspace_regions_are_disjoint_aligned_and_inside():
    for M, K, N, r in [(9437, 5120, 15360, 384), (1, 64, 128, 16), (200, 256, 384, 0), (37726, 13824, 5120, 128)]:
        st, off = h3lin.h3lin_forward_workspace_regions(M, K, N, r)
        assert st == h3lin.H3LIN_OK
        codes, scales, u, b, ts, status = off
        total = h3lin.h3lin_forward_workspace_bytes(M, K, N, r)
        assert (ts, status) == (4, 0)
        assert h3lin.h3lin_quant_workspace_bytes() <= codes
        ends = [(codes, codes + M * K // 2), (scales, scales + h3lin.h3lin_scales_bytes(M, K)),
                (u, u + M * r * 2), (b, b + N * r * 2)]
        for (lo, hi), (lo2, _) in zip(ends, ends[1:]):
            assert hi <= lo2
        assert ends[-1][1] <= total
        assert all(o % 1024 == 0 for o in (codes, scales, u, b))
    assert h3lin.h3lin_forward_workspace_regions(10, 100, 128, 16)[0] == h3lin.H3LIN_E_SHAPE
    assert h3lin.lib().h3lin_forward_workspace_regions(10, 64, 128, 16, None) == h3lin.H3LIN_E_INVALID


A = 0x10000  # an aligned fake device address (never dereferenced on error paths)


def _weight(N=384, K=256):
    return h3lin.h3lin_weight(A, A, A, N, K)


def _fwd(**kw):
    args = dict(x=A, M=200, pqs=None, weight=_weight(), epilogue=0, adapter=None, strength=1.0, out=A,
                out_dtype=0, ws=A, ws_bytes=1 << 30, stream=None)
    args.update(kw)
    return h3lin.h3lin_forward(args["x"], args["M"], args["pqs"], args["weight"], args["epilogue"],
                               args["adapter"], args["strength"], args["out"], args["out_dtype"], args["ws"],
                               args["ws_bytes"], args["stream"])


def test_forward_rejects_invalid_arguments():
    E = h3lin
    assert _fwd(x=None) == E.H3LIN_E_INVALID
    assert _fwd(out=None) == E.H3LIN_E_INVALID
    assert _fwd(weight=h3lin.h3lin_weight(None, A, A, 384, 256)) == E.H3LIN_E_INVALID
    assert _fwd(epilogue=7) == E.H3LIN_E_INVALID
    assert _fwd(out_dtype=2) == E.H3LIN_E_INVALID
    assert _fwd(strength=math.nan) == E.H3LIN_E_INVALID
    assert _fwd(strength=math.inf) == E.H3LIN_E_INVALID
    assert _fwd(M=-1) == E.H3LIN_E_SHAPE
    # no rows: valid, nothing enqueued, no buffer looked at (no device needed)
    assert _fwd(M=0, x=None, out=None, ws=None) == E.H3LIN_OK
    assert _fwd(M=0, weight=_weight(384, 200)) == E.H3LIN_E_SHAPE   # other rules still apply
    assert _fwd(weight=_weight(384, 200)) == E.H3LIN_E_SHAPE          # K % 64
    assert _fwd(weight=_weight(300, 256)) == E.H3LIN_E_SHAPE          # N % 128
    assert _fwd(weight=_weight(384, 256), epilogue=1) == E.H3LIN_E_SHAPE  # SiLU needs N % 256
    assert _fwd(x=A + 8) == E.H3LIN_E_ALIGN
    assert _fwd(out=A + 2) == E.H3LIN_E_ALIGN
    assert _fwd(pqs=A + 4) == E.H3LIN_E_ALIGN
    assert _fwd(ws_bytes=1024) == E.H3LIN_E_WORKSPACE


@pytest.mark.parametrize("rank,ok", [(16, True), (24, False), (128, True), (256, True), (272, False),
                                     (288, True), (384, True), (512, True), (544, False), (8, False), (0, False)])
def test_forward_rank_rule(rank, ok):
    ad = h3lin.h3lin_adapter(A, A, rank, float(rank))
    st = _fwd(adapter=ad)
    if ok:
        assert st not in (h3lin.H3LIN_E_SHAPE, h3lin.H3LIN_E_INVALID), st
    else:
        assert st == h3lin.H3LIN_E_SHAPE


def test_forward_adapter_checks():
    E = h3lin
    assert _fwd(adapter=h3lin.h3lin_adapter(None, A, 16, 16.0)) == E.H3LIN_E_INVALID
    assert _fwd(adapter=h3lin.h3lin_adapter(A, A, 16, math.nan)) == E.H3LIN_E_INVALID
    assert _fwd(adapter=h3lin.h3lin_adapter(A + 4, A, 16, 16.0)) == E.H3LIN_E_ALIGN
    # strength 0 selects the base path: the adapter is not even looked at
    bad = h3lin.h3lin_adapter(None, None, 3, math.nan)
    assert _fwd(adapter=bad, strength=0.0) not in (E.H3LIN_E_INVALID, E.H3LIN_E_SHAPE)


def test_quantize_rejects_invalid_arguments():
    E = h3lin
    q = lambda **kw: h3lin.h3lin_quantize_act(kw.get("x", A), kw.get("M", 10), kw.get("K", 64), kw.get("pqs"),
                                              kw.get("codes", A), kw.get("scales", A), kw.get("ts", A),
                                              kw.get("ws", A), kw.get("ws_bytes", 1 << 20), None)
    assert q(x=None) == E.H3LIN_E_INVALID
    assert q(ts=None) == E.H3LIN_E_INVALID
    assert q(K=96) == E.H3LIN_E_SHAPE
    assert q(M=-1) == E.H3LIN_E_SHAPE
    assert q(M=0, x=None, codes=None, scales=None, ts=None, ws=None) == E.H3LIN_OK
    assert q(codes=A + 1) == E.H3LIN_E_ALIGN
    assert q(ws_bytes=16) == E.H3LIN_E_WORKSPACE
    assert h3lin.h3lin_pack_weight(A, 0, 64, A, A, A, A, 1 << 20, None) == E.H3LIN_E_SHAPE


def test_merge_lora_rejects_invalid_arguments():
    E = h3lin
    ad = h3lin.h3lin_adapter(A, A, 16, 16.0)
    m = lambda **kw: h3lin.h3lin_merge_lora(kw.get("w", A), kw.get("N", 384), kw.get("K", 256), kw.get("pqs"),
                                            kw.get("adapter", ad), kw.get("strength", 1.0), kw.get("out", A), None)
    assert m(w=None) == E.H3LIN_E_INVALID
    assert m(out=None) == E.H3LIN_E_INVALID
    assert m(adapter=None) == E.H3LIN_E_INVALID
    assert m(adapter=h3lin.h3lin_adapter(A, None, 16, 16.0)) == E.H3LIN_E_INVALID
    assert m(adapter=h3lin.h3lin_adapter(A, A, 16, math.inf)) == E.H3LIN_E_INVALID
    assert m(strength=math.nan) == E.H3LIN_E_INVALID
    assert m(N=0) == E.H3LIN_E_SHAPE
    assert m(K=96) == E.H3LIN_E_SHAPE
    assert m(adapter=h3lin.h3lin_adapter(A, A, 24, 24.0)) == E.H3LIN_E_SHAPE
    assert m(w=A + 4) == E.H3LIN_E_ALIGN
    assert m(out=A + 2) == E.H3LIN_E_ALIGN
    assert m(pqs=A + 8) == E.H3LIN_E_ALIGN


def test_mlp_and_producer_argument_checks():
    E = h3lin
    gu, dn = _weight(1024, 256), _weight(384, 512)

    def mlp(**kw):
        a = dict(x=A, M=200, gu=gu, dn=dn, h=A, out=A, ws=A, ws_bytes=1 << 30)
        a.update(kw)
        return h3lin.h3lin_mlp_forward(a["x"], a["M"], None, a["gu"], None, 1.0, None, a["dn"], None, 1.0, a["h"],
                                       a["out"], 0, a["ws"], a["ws_bytes"], None)

    assert mlp(gu=None) == E.H3LIN_E_INVALID
    assert mlp(dn=_weight(384, 256)) == E.H3LIN_E_SHAPE       # down's K must be N_gate_up / 2
    assert mlp(M=-1) == E.H3LIN_E_SHAPE
    assert mlp(h=None) == E.H3LIN_E_INVALID
    assert mlp(h=A + 4) == E.H3LIN_E_ALIGN
    assert mlp(ws_bytes=4096) == E.H3LIN_E_WORKSPACE
    assert mlp(M=0, x=None, h=None, out=None, ws=None) == E.H3LIN_OK
    assert mlp(gu=_weight(1152, 256), dn=_weight(384, 576)) == E.H3LIN_E_SHAPE   # SiLU*up needs N % 256

    def produce(**kw):
        a = dict(M=200, w=gu, out=A, ws=A, ws_bytes=1 << 30, next_pqs=None, next_ws=A, next_bytes=1 << 20)
        a.update(kw)
        return h3lin.h3lin_forward_gemm_produce(a["M"], a["w"], 1, None, 1.0, a["out"], a["ws"], a["ws_bytes"],
                                                a["next_pqs"], a["next_ws"], a["next_bytes"], None)

    assert produce(next_ws=None) == E.H3LIN_E_INVALID
    assert produce(next_ws=A + 8) == E.H3LIN_E_ALIGN
    assert produce(next_pqs=A + 4) == E.H3LIN_E_ALIGN
    assert produce(next_bytes=64) == E.H3LIN_E_WORKSPACE
    assert produce(M=0, out=None, ws=None, next_ws=None) == E.H3LIN_OK
    assert produce(M=-3) == E.H3LIN_E_SHAPE
    assert h3lin.h3lin_forward_prepare_produced(A, -1, None, dn, None, 1.0, A, 1 << 30, None) == E.H3LIN_E_SHAPE
    assert h3lin.h3lin_forward_prepare_produced(None, 5, None, dn, None, 1.0, A, 1 << 30, None) == E.H3LIN_E_INVALID


def test_qk_norm_rope_argument_checks():
    E = h3lin

    def call(M=10, qkv=A, qg=A, kg=A, pos=A, ws=A, ws_bytes=1 << 20, **kw):
        prm = dict(heads=40, head_dim=128, rot_dims=96, axis_dims=(32, 32, 32), theta=10000.0, eps=1e-6)
        prm.update(kw)
        return h3lin.h3lin_qk_norm_rope(qkv, M, h3lin.rope_params(**prm), qg, kg, pos, ws, ws_bytes, None)

    assert h3lin.h3lin_qk_norm_rope(A, 10, None, A, A, A, A, 1 << 20, None) == E.H3LIN_E_INVALID
    assert call(head_dim=64) == E.H3LIN_E_SHAPE
    assert call(rot_dims=100, axis_dims=(34, 34, 32)) == E.H3LIN_E_SHAPE     # rot % 16
    assert call(rot_dims=144, axis_dims=(48, 48, 48)) == E.H3LIN_E_SHAPE     # rot > head_dim
    assert call(axis_dims=(32, 32, 30)) == E.H3LIN_E_SHAPE                   # sum != rot
    assert call(axis_dims=(31, 33, 32)) == E.H3LIN_E_SHAPE                   # odd axis
    assert call(heads=0) == E.H3LIN_E_SHAPE
    assert call(M=-1) == E.H3LIN_E_SHAPE
    assert call(theta=0.0) == E.H3LIN_E_INVALID
    assert call(eps=-1.0) == E.H3LIN_E_INVALID
    assert call(eps=math.nan) == E.H3LIN_E_INVALID
    assert call(M=0, qkv=None, qg=None, kg=None, pos=None, ws=None) == E.H3LIN_OK
    assert call(qkv=None) == E.H3LIN_E_INVALID
    assert call(qkv=A + 8) == E.H3LIN_E_ALIGN
    assert call(qg=A + 4) == E.H3LIN_E_ALIGN
    assert call(pos=A + 2) == E.H3LIN_E_ALIGN
    assert call(ws=None) == E.H3LIN_E_INVALID
    assert call(ws=A + 8) == E.H3LIN_E_ALIGN
    assert call(ws_bytes=64) == E.H3LIN_E_WORKSPACE


def test_forward_qk_rope_argument_checks():
    E = h3lin
    w = _weight(3 * 4 * 128, 256)   # 4 heads

    def full(M=10, x=A, w=w, qg=A, kg=A, pos=A, out=A, ws=A, ws_bytes=1 << 30, **kw):
        prm = dict(heads=4, head_dim=128, rot_dims=96, axis_dims=(32, 32, 32), theta=10000.0, eps=1e-6)
        prm.update(kw)
        return h3lin.h3lin_forward_qk_rope(x, M, None, w, None, 1.0, h3lin.rope_params(**prm), qg, kg, pos, out,
                                           ws, ws_bytes, None)

    def gemm(M=10, w=w, qg=A, kg=A, pos=A, out=A, ws=A, ws_bytes=1 << 30, **kw):
        prm = dict(heads=4, head_dim=128, rot_dims=96, axis_dims=(32, 32, 32), theta=10000.0, eps=1e-6)
        prm.update(kw)
        return h3lin.h3lin_forward_gemm_qk_rope(M, w, None, 1.0, h3lin.rope_params(**prm), qg, kg, pos, out, ws,
                                                ws_bytes, None)

    for call in (full, gemm):
        assert call(head_dim=64) == E.H3LIN_E_SHAPE
        assert call(axis_dims=(32, 32, 30)) == E.H3LIN_E_SHAPE
        assert call(theta=-1.0) == E.H3LIN_E_INVALID
        # valid parameters the fused epilogue does not serve
        assert call(rot_dims=64, axis_dims=(32, 16, 16)) == E.H3LIN_E_UNSUPPORTED
        assert call(heads=3, w=_weight(3 * 3 * 128, 256)) == E.H3LIN_E_UNSUPPORTED   # N % 256 != 0
        assert call(heads=5) == E.H3LIN_E_SHAPE                                     # N != 3 heads 128
        assert call(w=None) == E.H3LIN_E_INVALID
        assert call(M=-1) == E.H3LIN_E_SHAPE
        assert call(M=0, qg=None, kg=None, pos=None, out=None, ws=None) == E.H3LIN_OK
        assert call(qg=None) == E.H3LIN_E_INVALID
        assert call(pos=None) == E.H3LIN_E_INVALID
        assert call(kg=A + 4) == E.H3LIN_E_ALIGN
        assert call(pos=A + 2) == E.H3LIN_E_ALIGN
        assert call(out=None) == E.H3LIN_E_INVALID
        assert call(ws=A + 8) == E.H3LIN_E_ALIGN
    assert full(x=None) == E.H3LIN_E_INVALID
    # the workspace must hold h3lin_forward's regions plus M * 384 bytes of angles
    M, K, N = 1000, 256, 1536
    need = h3lin.h3lin_forward_qk_rope_workspace_bytes(M, K, N, 0)
    assert need >= h3lin.h3lin_forward_workspace_bytes(M, K, N, 0) + M * 48 * 8
    assert full(M=M, ws_bytes=need - 1) == E.H3LIN_E_WORKSPACE
    assert gemm(M=M, ws_bytes=need - 1) == E.H3LIN_E_WORKSPACE
    assert h3lin.h3lin_forward_qk_rope_workspace_bytes(-1, K, N, 0) == 0


def test_modulate_produce_argument_checks():
    E = h3lin

    def call(x=A, M=10, K=5120, table=A, T=3, rows=A, eps=1e-6, out=A, pqs=None, ws=A, ws_bytes=1 << 20):
        return h3lin.h3lin_modulate_produce(x, M, K, table, T, rows, eps, out, pqs, ws, ws_bytes, None)

    assert call(K=96) == E.H3LIN_E_SHAPE
    assert call(K=8256) == E.H3LIN_E_SHAPE
    assert call(T=0) == E.H3LIN_E_SHAPE
    assert call(M=-2) == E.H3LIN_E_SHAPE
    assert call(eps=math.inf) == E.H3LIN_E_INVALID
    assert call(M=0, x=None, table=None, rows=None, out=None, ws=None) == E.H3LIN_OK
    assert call(table=None) == E.H3LIN_E_INVALID
    assert call(ws=None) == E.H3LIN_E_INVALID
    assert call(out=A + 4) == E.H3LIN_E_ALIGN
    assert call(rows=A + 2) == E.H3LIN_E_ALIGN
    assert call(pqs=A + 8) == E.H3LIN_E_ALIGN
    assert call(ws_bytes=100) == E.H3LIN_E_WORKSPACE


def test_mlp_workspace_is_the_larger_projection_workspace():
    M, K, Ngu, Nd, r = 37726, 5120, 27648, 5120, 128
    want = max(h3lin.h3lin_forward_workspace_bytes(M, K, Ngu, r), h3lin.h3lin_forward_workspace_bytes(M, Ngu // 2, Nd, r))
    assert h3lin.h3lin_mlp_workspace_bytes(M, K, Ngu, Nd, r) == want
    assert h3lin.h3lin_mlp_workspace_bytes(M, K, 1000, Nd, r) == 0      # gate/up rows % 256
    assert h3lin.h3lin_mlp_workspace_bytes(-1, K, Ngu, Nd, r) == 0


@pytest.mark.skipif(__import__("tests._util", fromlist=["have_gpu"]).have_gpu(), reason="GPU present")
def test_valid_call_without_gpu_reports_cuda_error():
    # every host check passes; the call then fails to find a device and says so
    assert _fwd() in (h3lin.H3LIN_E_CUDA, h3lin.H3LIN_E_UNSUPPORTED)


def test_native_scale_layout_is_a_bijection():
    from tests._util import native_scale_offsets
    for rows, K in [(128, 64), (200, 256), (300, 320)]:
        off = native_scale_offsets(rows, K).reshape(-1)
        assert len(set(off.tolist())) == off.size
        assert off.max() < h3lin.h3lin_scales_bytes(rows, K)


def test_noalloc_host_checks():
    # the allocation-free forward refuses work beyond its fixed scratch, and a
    # missing weight, on the host: before it looks up any device
    K, N = 5120, 15360
    M = 1 + h3lin.H3LIN_NOALLOC_SCRATCH_BYTES // (K // 2)
    w = h3lin.h3lin_weight(A, A, A, N, K)
    assert h3lin.h3lin_forward_noalloc(A, M, None, w, 0, None, 1.0, A, 0, None) == h3lin.H3LIN_E_WORKSPACE
    assert h3lin.h3lin_forward_noalloc(A, 16, None, None, 0, None, 1.0, A, 0, None) == h3lin.H3LIN_E_INVALID
    # its status read needs somewhere to put the word (checked before any device call)
    assert h3lin.lib().h3lin_noalloc_read_status(None, None) == h3lin.H3LIN_E_INVALID
    # the projection the GPU test of this entry point runs fits in the scratch
    fits = h3lin.h3lin_forward_workspace_bytes(1024, 1024, 1280, 128)
    assert 0 < fits <= h3lin.H3LIN_NOALLOC_SCRATCH_BYTES


def test_bounds_build_links_exports_and_reports_itself():
    """The bounds-checked build compiles, exports every declared entry point
    and says it is the bounds build; the normal build refuses the bounds
    self-test on the host, before touching any device."""
    import subprocess
    import sys
    from nvfp4_linear_lora_gb300 import build as h3build
    path = h3build.build(bounds=True)
    assert os.path.exists(path)
    code = ("import ctypes; L = ctypes.CDLL(%r); "
            "names = %r; missing = [n for n in names if not hasattr(L, n)]; "
            "assert not missing, missing; print(L.h3lin_bounds_build())") % (path, _declared_functions())
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "1", r.stdout + r.stderr
    assert h3lin.h3lin_bounds_build() == 0
    assert h3lin.h3lin_selftest_bounds(A, 1 << 20, None) == h3lin.H3LIN_E_UNSUPPORTED
    assert h3lin.h3lin_status_string(h3lin.H3LIN_E_BOUNDS).startswith("a kernel index")
