"""Float64 CPU oracle (test infrastructure; not part of the product path).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference legs may import this package.  It is independent of the
CUDA library: neither imports the other and they share no code.

Modules: ``attention`` (masked attention, TileAttention partial states, the
LSE merge, the online recurrence, gradients, the sliding-window band),
``partition`` (zigzag, packed and striped splits), ``ring`` (the ring walk
over logical ranks, forward and backward), ``rope`` (rotary position
embedding at zigzag / THD positions), ``hybrid`` (the per-sub-sequence CP
schedule and the token layout of one round).
Every function is pinned by ``tests/test_oracle_*.py``.
"""

from . import attention, hybrid, partition, ring, rope  # noqa: F401
