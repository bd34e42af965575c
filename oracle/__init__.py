"""CPU oracle (test infrastructure only): fp64 quantiser, packer, dequantise-then-matvec.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package.  The library never does.
"""
from .q4_oracle import *  # noqa: F401,F403
from .q4_oracle import GROUP, LEVELS, QuantiseRangeError  # noqa: F401
