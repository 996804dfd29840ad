"""fp64 CPU oracle for decode-step KV page retrieval (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path (the CUDA library and its
Python binding) never does.
"""
from .oracle import *  # noqa: F401,F403
