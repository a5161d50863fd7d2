"""GB300-native dynamic-LoRA NVFP4 linear.

``h3lin`` is the thin ctypes binding of the C-ABI library ``libh3lin.so``
(built in-tree from ``csrc/`` by ``build.py``); ``synth`` draws the seeded
synthetic inputs and ``configs`` names the workloads.  Importing the package
does not load the library; the first call into ``h3lin`` does, and fails
loudly when it is missing.
"""
