"""CPU oracle for the DFlash draft step — test infrastructure, not part of the product.

Only the tests, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`
import this package. The CUDA library never calls it and shares no code with it.
"""
from .dflash_oracle import *  # noqa: F401,F403
