"""Plain fp64 CPU oracle for indexer-driven sparse attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs use it. It shares no code, header, table or helper with the CUDA
library in ``indexer_driven_sparse_gb300``; the two meet only through the seeded
input generators, which hold none of the method's arithmetic.
"""

from .qsa_oracle import *  # noqa: F401,F403
