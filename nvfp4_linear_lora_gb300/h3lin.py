"""Thin ctypes binding of ``libh3lin.so`` (C ABI declared in ``include/h3lin.h``).

The ``h3lin_*`` functions mirror the C entry points one to one (plain
integers for device pointers and streams).  The torch helpers below them only
marshal arguments: they allocate buffers with torch, pass ``data_ptr()`` and
the current stream, and raise on a non-zero status.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback — a
missing library raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
# H3LIN_BOUNDS=1 loads the bounds-checked build (libh3lin_bounds.so: every
# plain global index checked in the kernels, a bad one reported in the
# workspace status word as H3LIN_E_BOUNDS instead of touching memory).
BOUNDS = os.environ.get("H3LIN_BOUNDS") == "1"
LIB_PATH = os.path.join(_HERE, "libh3lin_bounds.so" if BOUNDS else "libh3lin.so")
# H3LIN_CANARY=1 gives every workspace and output the helpers below allocate a
# guard region of CANARY_BYTES filled with CANARY_BYTE right after it;
# check_canaries() verifies that no kernel wrote past a buffer's end.
CANARY = os.environ.get("H3LIN_CANARY") == "1"
CANARY_BYTES = 4096
CANARY_BYTE = 0xA5

H3LIN_OK = 0
H3LIN_E_INVALID = 1
H3LIN_E_SHAPE = 2
H3LIN_E_ALIGN = 3
H3LIN_E_WORKSPACE = 4
H3LIN_E_CUDA = 5
H3LIN_E_TIMEOUT = 6
H3LIN_E_UNSUPPORTED = 7
H3LIN_E_BOUNDS = 8
H3LIN_OUT_BF16 = 0
H3LIN_OUT_F32 = 1
H3LIN_EPI_NONE = 0
H3LIN_EPI_SILU_MUL = 1


class H3linError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: status {status} ({h3lin_status_string(status)})")


class h3lin_weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class h3lin_adapter(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("rank", ctypes.c_int32),
                ("alpha", ctypes.c_float)]


class h3lin_rope_params(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("rot_dims", ctypes.c_int32),
                ("axis_dims", ctypes.c_int32 * 3), ("theta", ctypes.c_float), ("eps", ctypes.c_float)]


_lib = None
_vp, _i64, _i32, _sz, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float

_SIGNATURES = {
    "h3lin_abi_version": (_i32, []),
    "h3lin_status_string": (ctypes.c_char_p, [_i32]),
    "h3lin_codes_bytes": (_sz, [_i64, _i64]),
    "h3lin_scales_bytes": (_sz, [_i64, _i64]),
    "h3lin_quant_workspace_bytes": (_sz, []),
    "h3lin_forward_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32]),
    "h3lin_workspace_init": (_i32, [_vp, _sz, _vp]),
    "h3lin_forward_workspace_regions": (_i32, [_i64, _i64, _i64, _i32, ctypes.POINTER(_sz)]),
    "h3lin_quantize_act": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "h3lin_pack_weight": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "h3lin_forward": (_i32, [_vp, _i64, _vp, ctypes.POINTER(h3lin_weight), _i32, ctypes.POINTER(h3lin_adapter),
                             _f32, _vp, _i32, _vp, _sz, _vp]),
    "h3lin_forward_prepare": (_i32, [_vp, _i64, _vp, ctypes.POINTER(h3lin_weight), ctypes.POINTER(h3lin_adapter),
                                     _f32, _vp, _sz, _vp]),
    "h3lin_forward_gemm": (_i32, [_i64, ctypes.POINTER(h3lin_weight), _i32, ctypes.POINTER(h3lin_adapter), _f32,
                                  _vp, _i32, _vp, _sz, _vp]),
    "h3lin_forward_gemm_produce": (_i32, [_i64, ctypes.POINTER(h3lin_weight), _i32, ctypes.POINTER(h3lin_adapter),
                                          _f32, _vp, _vp, _sz, _vp, _vp, _sz, _vp]),
    "h3lin_forward_prepare_produced": (_i32, [_vp, _i64, _vp, ctypes.POINTER(h3lin_weight),
                                              ctypes.POINTER(h3lin_adapter), _f32, _vp, _sz, _vp]),
    "h3lin_mlp_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _i32]),
    "h3lin_mlp_forward": (_i32, [_vp, _i64, _vp, ctypes.POINTER(h3lin_weight), ctypes.POINTER(h3lin_adapter), _f32,
                                 _vp, ctypes.POINTER(h3lin_weight), ctypes.POINTER(h3lin_adapter), _f32,
                                 _vp, _vp, _i32, _vp, _sz, _vp]),
    "h3lin_qk_norm_rope": (_i32, [_vp, _i64, ctypes.POINTER(h3lin_rope_params), _vp, _vp, _vp, _vp, _sz, _vp]),
    "h3lin_forward_qk_rope_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32]),
    "h3lin_forward_qk_rope": (_i32, [_vp, _i64, _vp, ctypes.POINTER(h3lin_weight), ctypes.POINTER(h3lin_adapter),
                                     _f32, ctypes.POINTER(h3lin_rope_params), _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "h3lin_forward_gemm_qk_rope": (_i32, [_i64, ctypes.POINTER(h3lin_weight), ctypes.POINTER(h3lin_adapter), _f32,
                                          ctypes.POINTER(h3lin_rope_params), _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "h3lin_modulate_produce": (_i32, [_vp, _i64, _i64, _vp, _i32, _vp, _f32, _vp, _vp, _vp, _sz, _vp]),
    "h3lin_read_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32)]),
    "h3lin_selftest_wait_timeout": (_i32, [_vp, _sz, _i64, _vp]),
    "h3lin_selftest_bounds": (_i32, [_vp, _sz, _vp]),
    "h3lin_bounds_build": (_i32, []),
    "h3lin_merge_lora": (_i32, [_vp, _i64, _i64, _vp, ctypes.POINTER(h3lin_adapter), _f32, _vp, _vp]),
    "h3lin_forward_noalloc": (_i32, [_vp, _i64, _vp, ctypes.POINTER(h3lin_weight), _i32,
                                     ctypes.POINTER(h3lin_adapter), _f32, _vp, _i32, _vp]),
    "h3lin_noalloc_read_status": (_i32, [_vp, ctypes.POINTER(_i32)]),
}

H3LIN_NOALLOC_SCRATCH_BYTES = 64 << 20


def lib():
    """Load ``libh3lin.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with nvfp4_linear_lora_gb300.build.build()"
                               + (" (bounds=True)" if BOUNDS else ""))
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


# ----------------------------------------------------------- C entry points
def h3lin_abi_version():
    return lib().h3lin_abi_version()


def h3lin_status_string(status):
    return lib().h3lin_status_string(int(status)).decode()


def h3lin_codes_bytes(rows, K):
    return lib().h3lin_codes_bytes(rows, K)


def h3lin_scales_bytes(rows, K):
    return lib().h3lin_scales_bytes(rows, K)


def h3lin_quant_workspace_bytes():
    return lib().h3lin_quant_workspace_bytes()


def h3lin_forward_workspace_bytes(M, K, N, max_rank):
    return lib().h3lin_forward_workspace_bytes(M, K, N, max_rank)


def h3lin_forward_workspace_regions(M, K, N, rank):
    """(status, [codes, scales, u, B', ts_x, status word] byte offsets)."""
    off = (_sz * 6)()
    st = lib().h3lin_forward_workspace_regions(M, K, N, rank, off)
    return st, list(off)


def h3lin_workspace_init(ws, ws_bytes, stream):
    return lib().h3lin_workspace_init(ws, ws_bytes, stream)


def h3lin_quantize_act(x, M, K, pqs, codes, scales, tensor_scale, ws, ws_bytes, stream):
    return lib().h3lin_quantize_act(x, M, K, pqs, codes, scales, tensor_scale, ws, ws_bytes, stream)


def h3lin_pack_weight(w, N, K, codes, scales, tensor_scale, ws, ws_bytes, stream):
    return lib().h3lin_pack_weight(w, N, K, codes, scales, tensor_scale, ws, ws_bytes, stream)


def h3lin_forward(x, M, pqs, weight, epilogue, adapter, strength, out, out_dtype, ws, ws_bytes, stream):
    wp = ctypes.byref(weight) if weight is not None else None
    ap = ctypes.byref(adapter) if adapter is not None else None
    return lib().h3lin_forward(x, M, pqs, wp, epilogue, ap, strength, out, out_dtype, ws, ws_bytes, stream)


def h3lin_forward_prepare(x, M, pqs, weight, adapter, strength, ws, ws_bytes, stream):
    wp = ctypes.byref(weight) if weight is not None else None
    ap = ctypes.byref(adapter) if adapter is not None else None
    return lib().h3lin_forward_prepare(x, M, pqs, wp, ap, strength, ws, ws_bytes, stream)


def h3lin_forward_gemm(M, weight, epilogue, adapter, strength, out, out_dtype, ws, ws_bytes, stream):
    wp = ctypes.byref(weight) if weight is not None else None
    ap = ctypes.byref(adapter) if adapter is not None else None
    return lib().h3lin_forward_gemm(M, wp, epilogue, ap, strength, out, out_dtype, ws, ws_bytes, stream)


def _ref(s):
    return ctypes.byref(s) if s is not None else None


def h3lin_forward_gemm_produce(M, weight, epilogue, adapter, strength, out, ws, ws_bytes, next_pqs, next_ws,
                               next_ws_bytes, stream):
    return lib().h3lin_forward_gemm_produce(M, _ref(weight), epilogue, _ref(adapter), strength, out, ws, ws_bytes,
                                            next_pqs, next_ws, next_ws_bytes, stream)


def h3lin_forward_prepare_produced(x, M, pqs, weight, adapter, strength, ws, ws_bytes, stream):
    return lib().h3lin_forward_prepare_produced(x, M, pqs, _ref(weight), _ref(adapter), strength, ws, ws_bytes,
                                                stream)


def h3lin_mlp_workspace_bytes(M, K, N_gate_up, N_down, max_rank):
    return lib().h3lin_mlp_workspace_bytes(M, K, N_gate_up, N_down, max_rank)


def h3lin_mlp_forward(x, M, gu_pqs, gate_up, gu_adapter, gu_strength, down_pqs, down, down_adapter, down_strength,
                      h, out, out_dtype, ws, ws_bytes, stream):
    return lib().h3lin_mlp_forward(x, M, gu_pqs, _ref(gate_up), _ref(gu_adapter), gu_strength, down_pqs,
                                   _ref(down), _ref(down_adapter), down_strength, h, out, out_dtype, ws, ws_bytes,
                                   stream)


def h3lin_qk_norm_rope(qkv, M, params, q_gain, k_gain, positions, ws, ws_bytes, stream):
    return lib().h3lin_qk_norm_rope(qkv, M, _ref(params), q_gain, k_gain, positions, ws, ws_bytes, stream)


def h3lin_forward_qk_rope_workspace_bytes(M, K, N, max_rank):
    return lib().h3lin_forward_qk_rope_workspace_bytes(M, K, N, max_rank)


def h3lin_forward_qk_rope(x, M, pqs, weight, adapter, strength, params, q_gain, k_gain, positions, out, ws, ws_bytes,
                          stream):
    return lib().h3lin_forward_qk_rope(x, M, pqs, _ref(weight), _ref(adapter), strength, _ref(params), q_gain,
                                       k_gain, positions, out, ws, ws_bytes, stream)


def h3lin_forward_gemm_qk_rope(M, weight, adapter, strength, params, q_gain, k_gain, positions, out, ws, ws_bytes,
                               stream):
    return lib().h3lin_forward_gemm_qk_rope(M, _ref(weight), _ref(adapter), strength, _ref(params), q_gain, k_gain,
                                            positions, out, ws, ws_bytes, stream)


def h3lin_modulate_produce(x, M, K, table, table_rows, row_table, eps, x_mod, next_pqs, next_ws, next_ws_bytes,
                           stream):
    return lib().h3lin_modulate_produce(x, M, K, table, table_rows, row_table, eps, x_mod, next_pqs, next_ws,
                                        next_ws_bytes, stream)


def h3lin_forward_noalloc(x, M, pqs, weight, epilogue, adapter, strength, out, out_dtype, stream):
    """h3lin_forward for callers that cannot allocate: the scratch is a fixed
    array inside the library (see include/h3lin.h for the rules)."""
    wp = ctypes.byref(weight) if weight is not None else None
    ap = ctypes.byref(adapter) if adapter is not None else None
    return lib().h3lin_forward_noalloc(x, M, pqs, wp, epilogue, ap, strength, out, out_dtype, stream)


def h3lin_noalloc_read_status(stream):
    """(call status, device status word of the allocation-free scratch); a set
    word is cleared by the read."""
    v = _i32(-1)
    st = lib().h3lin_noalloc_read_status(stream, ctypes.byref(v))
    return st, v.value


def h3lin_merge_lora(w, N, K, pqs, adapter, strength, w_out, stream):
    ap = ctypes.byref(adapter) if adapter is not None else None
    return lib().h3lin_merge_lora(w, N, K, pqs, ap, strength, w_out, stream)


def h3lin_selftest_wait_timeout(ws, ws_bytes, wait_cycles, stream):
    return lib().h3lin_selftest_wait_timeout(ws, ws_bytes, wait_cycles, stream)


def h3lin_selftest_bounds(ws, ws_bytes, stream):
    return lib().h3lin_selftest_bounds(ws, ws_bytes, stream)


def h3lin_bounds_build():
    return lib().h3lin_bounds_build()


def h3lin_read_status(ws, stream):
    v = _i32(-1)
    st = lib().h3lin_read_status(ws, stream, ctypes.byref(v))
    return st, v.value


# ------------------------------------------------------- torch marshalling
def _torch():
    import torch
    return torch


def _stream():
    return _torch().cuda.current_stream().cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(status, where):
    if status != H3LIN_OK:
        raise H3linError(status, where)


@dataclass
class PackedWeight:
    """NVFP4 weight owned by torch tensors: codes u8 [N, K/2], native scales,
    fp32 tensor scale (device)."""
    codes: object
    scales: object
    tensor_scale: object
    N: int
    K: int

    def c_struct(self):
        return h3lin_weight(self.codes.data_ptr(), self.scales.data_ptr(), self.tensor_scale.data_ptr(),
                            self.N, self.K)


@dataclass
class Adapter:
    """A resident LoRA adapter: A bf16 [rank, K], B bf16 [N, rank] on the device."""
    A: object
    B: object
    rank: int
    alpha: float

    def c_struct(self):
        return h3lin_adapter(self.A.data_ptr(), self.B.data_ptr(), self.rank, self.alpha)


_guards = []   # (guard tensor, where) of the buffers allocated with a canary tail


def _alloc(shape, dtype, device):
    """torch.empty, or (with H3LIN_CANARY=1) a view of a larger buffer whose
    CANARY_BYTES-long tail is filled with CANARY_BYTE and remembered."""
    torch = _torch()
    if not CANARY:
        return torch.empty(shape, dtype=dtype, device=device)
    n = 1
    for d in shape:
        n *= int(d)
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    raw = torch.empty(nbytes + CANARY_BYTES, dtype=torch.uint8, device=device)
    raw[nbytes:].fill_(CANARY_BYTE)
    _guards.append((raw[nbytes:], f"{tuple(shape)} {dtype}"))
    return raw[:nbytes].view(dtype).view(shape)


def check_canaries():
    """Raise if a kernel wrote into the guard tail of any buffer allocated
    since the last check (H3LIN_CANARY=1 only); forget those buffers."""
    global _guards
    if not CANARY:
        return
    torch = _torch()
    torch.cuda.synchronize()
    bad = [where for g, where in _guards if not bool((g == CANARY_BYTE).all())]
    _guards = []
    if bad:
        raise AssertionError(f"canary overwritten after: {bad}")


_bounds_ws = []   # bounds build: the workspaces whose status words check_bounds_status() reads


def check_bounds_status():
    """Bounds build only: raise if any workspace allocated since the last check
    recorded H3LIN_E_BOUNDS (a kernel index left its buffer); forget them."""
    global _bounds_ws
    if not BOUNDS:
        return
    torch = _torch()
    torch.cuda.synchronize()
    hit = [int(w.numel()) for w in _bounds_ws
           if int(w[:4].view(torch.int32).item()) == H3LIN_E_BOUNDS]
    _bounds_ws = []
    if hit:
        raise AssertionError(f"H3LIN_E_BOUNDS recorded in workspaces of {hit} bytes")


def new_workspace(nbytes, device="cuda"):
    torch = _torch()
    ws = _alloc((int(nbytes),), torch.uint8, device)
    if BOUNDS:
        _bounds_ws.append(ws)
    _check(h3lin_workspace_init(ws.data_ptr(), ws.numel(), _stream()), "h3lin_workspace_init")
    return ws


def quantize_act(x, pre_quant_scale=None, workspace=None):
    """x bf16 [M, K] (cuda) -> (codes u8 [M, K/2], native scales u8, tensor scale f32 [1])."""
    torch = _torch()
    M, K = x.shape
    codes = _alloc((M, K // 2), torch.uint8, x.device)
    scales = _alloc((h3lin_scales_bytes(M, K),), torch.uint8, x.device)
    ts = _alloc((1,), torch.float32, x.device)
    ws = workspace if workspace is not None else new_workspace(h3lin_quant_workspace_bytes(), x.device)
    _check(h3lin_quantize_act(x.data_ptr(), M, K, _ptr(pre_quant_scale), codes.data_ptr(), scales.data_ptr(),
                              ts.data_ptr(), ws.data_ptr(), ws.numel(), _stream()), "h3lin_quantize_act")
    return codes, scales, ts


def pack_weight(w, workspace=None):
    """w bf16 [N, K] (cuda) -> PackedWeight."""
    torch = _torch()
    N, K = w.shape
    codes = _alloc((N, K // 2), torch.uint8, w.device)
    scales = _alloc((h3lin_scales_bytes(N, K),), torch.uint8, w.device)
    ts = _alloc((1,), torch.float32, w.device)
    ws = workspace if workspace is not None else new_workspace(h3lin_quant_workspace_bytes(), w.device)
    _check(h3lin_pack_weight(w.data_ptr(), N, K, codes.data_ptr(), scales.data_ptr(), ts.data_ptr(),
                             ws.data_ptr(), ws.numel(), _stream()), "h3lin_pack_weight")
    return PackedWeight(codes, scales, ts, N, K)


def forward(x, weight, pre_quant_scale=None, adapter=None, strength=1.0, silu_mul=False, out=None,
            workspace=None, out_dtype=None):
    """One projection through ``h3lin_forward``; returns ``out`` (bf16 unless
    ``out_dtype``/``out`` say float32)."""
    torch = _torch()
    M = x.shape[0]
    n_out = weight.N // 2 if silu_mul else weight.N
    if out is None:
        out = _alloc((M, n_out), out_dtype or torch.bfloat16, x.device)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    code = H3LIN_OUT_F32 if out.dtype == torch.float32 else H3LIN_OUT_BF16
    if workspace is None:
        workspace = new_workspace(h3lin_forward_workspace_bytes(M, weight.K, weight.N,
                                                                adapter.rank if adapter else 0), x.device)
    wc = weight.c_struct()
    ac = adapter.c_struct() if adapter is not None else None
    _check(h3lin_forward(x.data_ptr(), M, _ptr(pre_quant_scale), wc,
                         H3LIN_EPI_SILU_MUL if silu_mul else H3LIN_EPI_NONE, ac, float(strength),
                         out.data_ptr(), code, workspace.data_ptr(), workspace.numel(), _stream()), "h3lin_forward")
    return out


def mlp_forward(x, gate_up, down, gate_up_pre_quant_scale=None, down_pre_quant_scale=None, gate_up_adapter=None,
                down_adapter=None, gate_up_strength=1.0, down_strength=1.0, h=None, out=None, out_dtype=None,
                workspace=None):
    """The MLP ``down(silu(gate(x)) * up(x))`` through ``h3lin_mlp_forward``
    (producer fusion: gate/up's epilogue reduces the amax of h for down's
    quantiser).  Returns ``(h, out)``; h is bf16 [M, N_gu/2]."""
    torch = _torch()
    M = x.shape[0]
    if h is None:
        h = _alloc((M, gate_up.N // 2), torch.bfloat16, x.device)
    if out is None:
        out = _alloc((M, down.N), out_dtype or torch.bfloat16, x.device)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    code = H3LIN_OUT_F32 if out.dtype == torch.float32 else H3LIN_OUT_BF16
    if workspace is None:
        r = max(gate_up_adapter.rank if gate_up_adapter else 0, down_adapter.rank if down_adapter else 0)
        workspace = new_workspace(h3lin_mlp_workspace_bytes(M, gate_up.K, gate_up.N, down.N, r), x.device)
    _check(h3lin_mlp_forward(x.data_ptr(), M, _ptr(gate_up_pre_quant_scale), gate_up.c_struct(),
                             gate_up_adapter.c_struct() if gate_up_adapter else None, float(gate_up_strength),
                             _ptr(down_pre_quant_scale), down.c_struct(),
                             down_adapter.c_struct() if down_adapter else None, float(down_strength),
                             h.data_ptr(), out.data_ptr(), code, workspace.data_ptr(), workspace.numel(),
                             _stream()), "h3lin_mlp_forward")
    return h, out


def rope_params(heads, head_dim=128, rot_dims=96, axis_dims=(32, 32, 32), theta=10000.0, eps=1e-6):
    return h3lin_rope_params(heads, head_dim, rot_dims, (ctypes.c_int32 * 3)(*axis_dims), theta, eps)


def qk_norm_rope(qkv, q_gain, k_gain, positions, heads, rot_dims=96, axis_dims=(32, 32, 32), theta=10000.0,
                 eps=1e-6, workspace=None):
    """In place on ``qkv`` bf16 [M, 3 * heads * 128]: per-head RMSNorm of Q and K
    (gains fp32 [128]) and split-half three-axis RoPE from ``positions`` int32
    [M, 3]; returns ``qkv``."""
    torch = _torch()
    if qkv.dtype != torch.bfloat16 or qkv.dim() != 2 or not qkv.is_contiguous():
        raise TypeError("qkv must be a contiguous 2-D bfloat16 tensor")
    if positions.dtype != torch.int32:
        raise TypeError("positions must be int32 [M, 3]")
    p = rope_params(heads, 128, rot_dims, axis_dims, theta, eps)
    ws = workspace if workspace is not None else new_workspace(h3lin_quant_workspace_bytes(), qkv.device)
    _check(h3lin_qk_norm_rope(qkv.data_ptr(), qkv.shape[0], p, q_gain.data_ptr(), k_gain.data_ptr(),
                              positions.data_ptr(), ws.data_ptr(), ws.numel(), _stream()), "h3lin_qk_norm_rope")
    return qkv


def forward_qk_rope(x, weight, q_gain, k_gain, positions, heads, pre_quant_scale=None, adapter=None, strength=1.0,
                    rot_dims=96, axis_dims=(32, 32, 32), theta=10000.0, eps=1e-6, out=None, workspace=None):
    """The QKV projection with Q/K RMSNorm + split-half RoPE in its epilogue
    (``h3lin_forward_qk_rope``): the same bf16 [M, 3 * heads * 128] as
    ``forward`` followed by ``qk_norm_rope``, in one GEMM."""
    torch = _torch()
    M = x.shape[0]
    if positions.dtype != torch.int32:
        raise TypeError("positions must be int32 [M, 3]")
    if out is None:
        out = _alloc((M, weight.N), torch.bfloat16, x.device)
    if out.dtype != torch.bfloat16:
        raise TypeError("out must be bfloat16")
    if workspace is None:
        workspace = new_workspace(h3lin_forward_qk_rope_workspace_bytes(M, weight.K, weight.N,
                                                                        adapter.rank if adapter else 0), x.device)
    p = rope_params(heads, 128, rot_dims, axis_dims, theta, eps)
    _check(h3lin_forward_qk_rope(x.data_ptr(), M, _ptr(pre_quant_scale), weight.c_struct(),
                                 adapter.c_struct() if adapter is not None else None, float(strength), p,
                                 q_gain.data_ptr(), k_gain.data_ptr(), positions.data_ptr(), out.data_ptr(),
                                 workspace.data_ptr(), workspace.numel(), _stream()), "h3lin_forward_qk_rope")
    return out


def modulate_produce(x, table, row_table, next_workspace, next_pre_quant_scale=None, eps=1e-6, out=None):
    """x_mod = bf16(LayerNorm(x) * (1 + scale) + shift) with the table row of each
    row (``table`` fp32 [T, 2, K], ``row_table`` int32 [M]); leaves the amax of
    |x_mod * next_pre_quant_scale| in ``next_workspace`` for
    ``h3lin_forward_prepare_produced``.  Returns x_mod (bf16 [M, K])."""
    torch = _torch()
    M, K = x.shape
    if out is None:
        out = _alloc((M, K), torch.bfloat16, x.device)
    _check(h3lin_modulate_produce(x.data_ptr(), M, K, table.data_ptr(), table.shape[0], row_table.data_ptr(),
                                  float(eps), out.data_ptr(), _ptr(next_pre_quant_scale), next_workspace.data_ptr(),
                                  next_workspace.numel(), _stream()), "h3lin_modulate_produce")
    return out


def forward_produced(x, weight, workspace, pre_quant_scale=None, adapter=None, strength=1.0, silu_mul=False,
                     out=None, out_dtype=None):
    """A projection whose input x was written by a producer (modulation or a
    producer GEMM) that left its amax in ``workspace``: prepare from those
    partials (one pass over x), then the GEMM.  Same result as ``forward``."""
    torch = _torch()
    M = x.shape[0]
    n_out = weight.N // 2 if silu_mul else weight.N
    if out is None:
        out = _alloc((M, n_out), out_dtype or torch.bfloat16, x.device)
    code = H3LIN_OUT_F32 if out.dtype == torch.float32 else H3LIN_OUT_BF16
    wc = weight.c_struct()
    ac = adapter.c_struct() if adapter is not None else None
    st = _stream()
    _check(h3lin_forward_prepare_produced(x.data_ptr(), M, _ptr(pre_quant_scale), wc, ac, float(strength),
                                          workspace.data_ptr(), workspace.numel(), st), "h3lin_forward_prepare_produced")
    _check(h3lin_forward_gemm(M, wc, H3LIN_EPI_SILU_MUL if silu_mul else H3LIN_EPI_NONE, ac, float(strength),
                              out.data_ptr(), code, workspace.data_ptr(), workspace.numel(), st), "h3lin_forward_gemm")
    return out


def merge_lora(w, adapter, strength=1.0, pre_quant_scale=None, out=None):
    """``bf16(w + strength * (alpha/rank) * B @ A / s)`` through ``h3lin_merge_lora``
    (s = ``pre_quant_scale``, 1 when None); ``out`` may be ``w`` itself (in place)."""
    torch = _torch()
    if w.dtype != torch.bfloat16 or w.dim() != 2:
        raise TypeError("w must be a 2-D bfloat16 tensor")
    if out is None:
        out = _alloc(tuple(w.shape), w.dtype, w.device)
    _check(h3lin_merge_lora(w.data_ptr(), w.shape[0], w.shape[1], _ptr(pre_quant_scale), adapter.c_struct(),
                            float(strength), out.data_ptr(), _stream()), "h3lin_merge_lora")
    return out


def read_status(workspace):
    st, v = h3lin_read_status(workspace.data_ptr(), _stream())
    _check(st, "h3lin_read_status")
    return v
