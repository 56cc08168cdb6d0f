"""CPU oracle for the W4A16 int4-weight linear layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (``w4a16_int4_weight_gb300``) never
imports it and shares no code with it.
"""

from .oracle import *  # noqa: F401,F403
