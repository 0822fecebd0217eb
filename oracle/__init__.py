"""CPU oracle for DSA sparse-attention decode (test infrastructure only).

A plain, slow, float64 restatement of what the decode path computes, written
from the method's description and shared with the CUDA library in nothing but
the seeded inputs of the ``workloads`` package.  Only the tests, the smoke
check of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it; the product path never does.
"""

from .dsa_oracle import *  # noqa: F401,F403
