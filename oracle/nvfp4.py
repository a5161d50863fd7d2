"""NVFP4 codec oracle: plain, slow, obviously-correct CPU reference.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` use it.  It shares no code with
the CUDA library and never imports the product package.

What is being encoded
---------------------
The pages name the format only as "NVFP4": the packed base weights of the
dynamic-LoRA linear (TURBO.md, h3-blackwell-runtime, section "Implementation")
and the "dynamic NVFP4 activation quantization" of the kernel path
(MiniMax-H3 Ultra Fast README, section "Kernel path", item 1; table "Active
optimization stack", rows Weights and Compute).  The encoding written out here
is the format's public definition, with the steps the pages leave open taken
in their plainest reading:

* element  : E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit), two
             codes per byte, even element in bits 0-3, odd element in bits 4-7;
* block    : one unsigned E4M3 scale per 16 consecutive elements along K;
* tensor   : one FP32 scale ``ts = amax / (6 * 448)`` per tensor (``ts = 1``
             when that quotient is zero).

Every floating-point step that decides a code is carried out in IEEE float32
with round-to-nearest-even, in exactly this order (so that the GPU kernels,
which take the same integer decisions in float32, can be compared bit for
bit):

1. ``v = x * s``                        pre_quant_scale ``s`` (absent -> 1)
2. ``amax = max |v|`` over the tensor, ``ts = amax / 2688`` (0 -> 1)
3. per 16-block: ``bamax = max |v|``; ``sb = E4M3_rne_sat(bamax / (6 * ts))``
4. ``d = decode(sb) * ts``
5. ``q = v / d`` (the IEEE float32 quotient); ``code = E2M1_rne_sat(q)`` with
   the sign of ``q`` kept (a negative value that rounds to zero gives code
   0x8).  A block with ``d == 0`` gets all-zero codes.

Step 5 is the plain definition of an element's code, the quotient of the
value by its block's dequantisation scale, rounded once to float32; nothing
on the pages asks for another order of operations.
"""
from __future__ import annotations

import numpy as np

# E2M1 magnitudes, indexed by the 3-bit magnitude code (exponent:mantissa).
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0
E4M3_MAX = 448.0
TENSOR_SCALE_DIVISOR = np.float32(6.0 * 448.0)  # 2688
BLOCK = 16


# --------------------------------------------------------------------------- E2M1
def e2m1_decode(codes) -> np.ndarray:
    """Decode 4-bit E2M1 codes (uint8 in 0..15) to float64 values."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = E2M1_VALUES[codes & 7]
    return np.where((codes & 8) != 0, -mag, mag)


def e2m1_encode(q) -> np.ndarray:
    """Round float32 values to E2M1 codes: nearest value, ties to the even code,
    magnitudes above 6 saturate to 6, the sign bit is the sign of ``q``.

    Within each binade the E2M1 values are equally spaced (0.5 below 2, 1 in
    [2, 4), 2 from 4), so rounding to nearest-even on the grid is rounding
    ``|q| / spacing`` to the nearest even integer; the even multiple is always
    the even code.  ``|q| / spacing`` is exact because the spacing is a power
    of two.
    """
    q = np.asarray(q, dtype=np.float32)
    a = np.abs(q).astype(np.float64)
    spacing = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.round(a / spacing) * spacing, E2M1_MAX)  # np.round: half to even
    mag_code = np.searchsorted(E2M1_VALUES, r).astype(np.uint8)
    assert np.all(E2M1_VALUES[mag_code] == r)
    sign = np.signbit(q).astype(np.uint8)
    return (mag_code | (sign << 3)).astype(np.uint8)


# --------------------------------------------------------------------------- E4M3
def e4m3_decode(bits) -> np.ndarray:
    """Decode E4M3 bit patterns (bias 7, subnormals, 0x7F/0xFF = NaN) to float64."""
    bits = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = (bits >> 7) & 1
    e = (bits >> 3) & 15
    m = bits & 7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    subnormal = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, subnormal, normal)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return np.where(s == 1, -val, val)


def e4m3_encode(y) -> np.ndarray:
    """Round float32 values to E4M3 bit patterns: nearest, ties to even,
    saturating to +-448 (the ``satfinite`` rule).  NaN inputs are rejected."""
    y = np.asarray(y, dtype=np.float32)
    assert not np.any(np.isnan(y)), "E4M3 encode: NaN input"
    a = np.abs(y).astype(np.float64)
    # floor(log2 a) from the exact binary exponent; subnormals share exponent -6
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e_unb = np.maximum(ex - 1, -6)
    spacing = np.exp2(e_unb - 3.0)  # 3 mantissa bits
    r = np.minimum(np.round(a / spacing) * spacing, E4M3_MAX)
    # re-encode the rounded magnitude (rounding may have carried into the next binade)
    _, ex2 = np.frexp(np.where(r > 0, r, 1.0))
    e2 = ex2 - 1
    is_sub = r < 2.0 ** -6
    m_sub = np.round(r / 2.0 ** -9)
    m_norm = np.round(r / np.exp2(e2 - 3.0)) - 8
    e_field = np.where(is_sub, 0, e2 + 7)
    m_field = np.where(is_sub, m_sub, m_norm)
    mag = (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    sign = np.signbit(y).astype(np.int64)
    out = (mag | (sign << 7)).astype(np.uint8)
    assert np.all(np.abs(e4m3_decode(out)) == r)
    return out


# --------------------------------------------------------------------------- quantiser
def prescale(x, pre_quant_scale=None) -> np.ndarray:
    """Step 1: ``v = x * s`` in float32 (x given as float32 holding bf16 values)."""
    x = np.asarray(x, dtype=np.float32)
    if pre_quant_scale is None:
        return x.copy()
    s = np.asarray(pre_quant_scale, dtype=np.float32)
    return x * s[None, :]


def tensor_amax(v) -> np.float32:
    """Step 2a: ``max |v|`` over the whole tensor (exact in float32)."""
    v = np.asarray(v, dtype=np.float32)
    return np.float32(np.max(np.abs(v))) if v.size else np.float32(0.0)


def tensor_scale(amax) -> np.float32:
    """Step 2b: ``ts = amax / 2688`` in float32; a zero quotient becomes 1."""
    ts = np.float32(amax) / TENSOR_SCALE_DIVISOR
    return np.float32(1.0) if ts == 0 else np.float32(ts)


def quantize_blocks(v, ts):
    """Steps 3-5 for rows of an already pre-scaled float32 matrix ``v [rows, K]``.

    Returns ``(codes [rows, K] uint8 unpacked, scales [rows, K/16] uint8)``.
    """
    v = np.asarray(v, dtype=np.float32)
    ts = np.float32(ts)
    rows, K = v.shape
    assert K % BLOCK == 0
    blk = v.reshape(rows, K // BLOCK, BLOCK)
    bamax = np.max(np.abs(blk), axis=2)                       # float32, exact
    six_ts = np.float32(6.0) * ts                              # float32 RN
    sb = e4m3_encode(bamax / six_ts)                           # float32 RN division
    d = e4m3_decode(sb).astype(np.float32) * ts                # float32 RN
    ok = d != 0
    with np.errstate(divide="ignore", invalid="ignore"):
        q = blk / np.where(ok, d, np.float32(1.0))[:, :, None]  # float32 RN division
    q = np.where(ok[:, :, None], q, np.float32(0.0)).astype(np.float32)
    codes = e2m1_encode(q)
    codes = np.where(ok[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    return codes.reshape(rows, K), sb


def pack_codes(codes) -> np.ndarray:
    """Two codes per byte: element 2j in bits 0-3, element 2j+1 in bits 4-7."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    out = np.empty((rows, 2 * half), dtype=np.uint8)
    out[:, 0::2] = packed & 15
    out[:, 1::2] = packed >> 4
    return out


def quantize(x, pre_quant_scale=None, rows=None, amax=None):
    """Full NVFP4 quantisation of ``x [M, K]`` (steps 1-5).

    ``rows`` (optional index array) restricts the returned codes/scales to those
    rows; the tensor scale is always taken over the whole tensor, or from
    ``amax`` when the caller already has it.

    Returns ``(packed codes [R, K/2] uint8, scales [R, K/16] uint8 row-major,
    tensor scale float32)``.
    """
    x = np.asarray(x, dtype=np.float32)
    if amax is None:
        amax = tensor_amax_chunked(x, pre_quant_scale)
    ts = tensor_scale(amax)
    sel = x if rows is None else x[np.asarray(rows)]
    codes, scales = quantize_blocks(prescale(sel, pre_quant_scale), ts)
    return pack_codes(codes), scales, ts


def tensor_amax_chunked(x, pre_quant_scale=None, chunk_rows=4096) -> np.float32:
    """``max |x * s|`` over the tensor, taken a slab of rows at a time."""
    x = np.asarray(x)
    m = np.float32(0.0)
    for r0 in range(0, x.shape[0], chunk_rows):
        m = max(m, tensor_amax(prescale(x[r0:r0 + chunk_rows], pre_quant_scale)))
    return np.float32(m)


def dequantize(packed, scales) -> np.ndarray:
    """``e2m1(code) * e4m3(scale)`` per element, float64, WITHOUT the tensor scale."""
    codes = unpack_codes(packed)
    rows, K = codes.shape
    vals = e2m1_decode(codes).reshape(rows, K // BLOCK, BLOCK)
    return (vals * e4m3_decode(scales)[:, :, None]).reshape(rows, K)
