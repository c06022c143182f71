"""KVarN CPU oracle -- test infrastructure only.

A plain double-precision C restatement of the KVarN group seal and of decode
attention over sealed groups (``kvarn_oracle.c``), loaded with ctypes, plus a
small Python model of the sink / sealed-groups / tail cache regions built on it.
Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. It shares no code with the CUDA library.
"""
from .oracle import *  # noqa: F401,F403
