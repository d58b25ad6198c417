"""CPU oracle of the two-level candidate indexer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package; the CUDA library never does.
"""
from . import ci_oracle  # noqa: F401
