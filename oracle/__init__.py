"""fp64 CPU oracle of the P-EAGLE draft pass (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / --impl reference
legs use this package.  The CUDA library never imports or calls it.
"""
from .peagle_oracle import *  # noqa: F401,F403
