"""CPU oracle of the routed-MoE feed-forward block (test infrastructure only).

Imported by the tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs
of ``bench.py``; never by the product package."""
from .moe_oracle import *  # noqa: F401,F403
