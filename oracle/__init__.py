"""CPU oracle for the indexer-Q preparation path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path never does.
"""
from . import iq_oracle  # noqa: F401
