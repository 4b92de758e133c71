"""CPU fp64 oracle of the DSpark draft-and-schedule step.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline legs of ``bench.py``; never by the product path.
"""
from .dspark_oracle import *  # noqa: F401,F403
from . import dspark_oracle  # noqa: F401
