"""GB300 (sm_103a) DSA sparse-attention decode.

The product is the C-ABI library ``libdsa_decode.so`` (header
``include/dsa_decode.h``); this package builds it (``build()``) and binds it
(``api``).  There is no other implementation: without the built library every
entry point raises.
"""

from ._build import LIB_PATH, build  # noqa: F401
from ._lib import lib  # noqa: F401

__all__ = ["build", "lib", "LIB_PATH"]
