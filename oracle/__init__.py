"""CPU oracle of the compressed-attention forward (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` use this package; the CUDA library never does.
"""
from . import v4_oracle  # noqa: F401
