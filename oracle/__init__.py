"""Float64 CPU oracle (test infrastructure; not part of the product path).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference legs may import this package.  It is independent of the
CUDA library: neither imports the other and they share no code.

Modules: ``attention`` (masked attention, TileAttention partial states, the
LSE merge, the online recurrence, gradients), ``partition`` (zigzag and
packed splits), ``ring`` (the ring walk over logical ranks, forward and
backward), ``rope`` (rotary position embedding at zigzag / THD positions).
Every function is pinned by ``tests/test_oracle_*.py``.
"""

from . import attention, partition, ring, rope  # noqa: F401
