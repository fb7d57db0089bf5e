"""Float64 CPU oracle for FusedKV attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product path never does.
"""
from .fusedkv_oracle import *  # noqa: F401,F403
