"""Writes ``nvfp4_tiny.txt``: the oracle's NVFP4 encoding of a small explicit
input, as a regression pin of the oracle.  Calls only ``oracle/``.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import nvfp4  # noqa: E402


def tiny_input():
    """Deterministic 4 x 64 activation and per-channel scale (no RNG)."""
    m = np.arange(4)[:, None]
    k = np.arange(64)[None, :]
    x = (((m * 37 + k * 11) % 29) - 14).astype(np.float32) / np.float32(3.5)
    x[2, 16:32] = 0.0
    x[3, 5] = np.float32(-40.0)
    x[1, 50] = np.float32(-1e-3)
    s = (0.5 + (np.arange(64) % 7) / 4.0).astype(np.float32)
    return x, s


def main():
    x, s = tiny_input()
    packed, scales, ts = nvfp4.quantize(x, s)
    lines = ["# oracle NVFP4 encoding of tests/golden/make_golden.py:tiny_input()",
             f"tensor_scale_f32_hex {np.float32(ts).view(np.uint32):08x}"]
    for r in range(packed.shape[0]):
        lines.append(f"scales_row{r} " + scales[r].tobytes().hex())
        lines.append(f"codes_row{r} " + packed[r].tobytes().hex())
    with open(os.path.join(HERE, "nvfp4_tiny.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
