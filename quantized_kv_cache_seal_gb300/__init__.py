"""KVarN on GB300: group seal (Hadamard rotation, 16 Sinkhorn iterations, round to
nearest, packing) and decode attention over sealed groups, as a C-ABI CUDA library
(``include/kvarn.h``, ``_build/libkvarn.so``) with a thin Python binding.

Method: fig1.dev "KVarN: Variance-Normalized KV-Cache Quantization Mitigates Error
Accumulation in Reasoning Tasks" ("What it is"); anbeeld.com "KVarN KV Cache:
Implementation and Benchmarks" (sections 1 and 2.1).
"""
from . import kvarn  # noqa: F401  (loads or builds libkvarn.so; fails loudly if it cannot)
from .kvarn import KVarNError  # noqa: F401
