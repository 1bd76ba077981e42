"""CPU oracle for the fused LM-head + Gumbel-max sampling path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The product library never imports
or links it, and it imports nothing from the product.
"""
from .oracle import *  # noqa: F401,F403
