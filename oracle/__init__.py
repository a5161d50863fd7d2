"""CPU oracle for the dynamic-LoRA NVFP4 linear.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline legs; never by the product package, whose
CUDA path shares no code with this one.  ``nvfp4`` holds the codec,
``linear`` the projection (base matmul, LoRA branch, SiLU*up).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, library routines (torch's E4M3 dtype, float64 matmul),
brute force on tiny inputs and the method's special cases.
"""
from . import nvfp4, linear  # noqa: F401
