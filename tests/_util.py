"""Test helpers: the native scale layout, parity metrics, GPU availability."""
import os

import numpy as np

# Parity bar for floating-point outputs (fixed by the workload definition):
MAX_REL_RMS = 3e-2      # max |gpu - oracle| / rms(oracle)
FRO_REL = 5e-3          # ||gpu - oracle||_F / ||oracle||_F


def native_scale_offsets(rows, K):
    """Byte offset of every (row, 16-block) scale in the library's native layout:
    512-byte atoms of 128 rows x 64 columns ordered [rows/128][K/64]; inside an
    atom row r, block j sits at (r % 32) * 16 + (r // 32) * 4 + j."""
    r = np.arange(rows)[:, None]
    j = np.arange(K // 16)[None, :]
    atom = (r // 128) * (K // 64) + j // 4
    rr = r % 128
    return atom * 512 + (rr % 32) * 16 + (rr // 32) * 4 + j % 4


def native_to_rowmajor(buf, rows, K):
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    return buf[native_scale_offsets(rows, K)]


def parity_metrics(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = gpu - ref
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(diff)) / rms), float(np.linalg.norm(diff) / np.linalg.norm(ref))


def assert_parity(gpu, ref, what=""):
    mx, fro = parity_metrics(gpu, ref)
    assert mx <= MAX_REL_RMS and fro <= FRO_REL, f"{what}: max/rms {mx:.3e} (<= {MAX_REL_RMS}), fro {fro:.3e} (<= {FRO_REL})"
    return mx, fro


def have_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
