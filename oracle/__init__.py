"""FP64 CPU oracle of the EXL3 linear layer (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.
"""
from .exl3_oracle import *  # noqa: F401,F403
