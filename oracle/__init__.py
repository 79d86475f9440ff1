"""CPU oracle for the multi-tenant LoRA delta (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does.
"""
from .oracle import *  # noqa: F401,F403
