"""Plain fp64 CPU oracle for the Ulysses attention layer (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path never does.
"""
from .ulysses_oracle import *  # noqa: F401,F403
