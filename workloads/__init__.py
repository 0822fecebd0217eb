"""Seeded synthetic inputs for DSA sparse-attention decode.

This package only draws random numbers and lays them out the way a paged
decode cache stores them (bf16 bits, fp8 e4m3 codes with a per-token fp32
scale, block tables, row positions).  It holds none of the decode method's
arithmetic: scoring, selection, attention and merging live in the library
(CUDA) and, independently, in the CPU oracle.  Both sides take their inputs
from here and from nowhere else.
"""

from .synth import (  # noqa: F401
    PagedCache,
    Spec,
    Workload,
    config_spec,
    make_workload,
    CONFIG_NAMES,
)
