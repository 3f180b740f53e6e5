"""CPU parity oracle for the gated W4 + low-rank compensated linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It is independent
of the CUDA library: it neither imports nor links anything from it.
"""
from .oracle import *  # noqa: F401,F403
