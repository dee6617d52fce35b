"""CPU oracle of the DFlash hot path -- TEST INFRASTRUCTURE, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it. It shares no code with the CUDA path.
"""
from .dflash_oracle import *  # noqa: F401,F403
from .dflash_oracle import (FLAG_ACCEPT_BOUNDARY, FLAG_CDF_BOUNDARY,  # noqa: F401
                            FLAG_DEGENERATE, FLAG_INVALID, FLAG_GATE_BOUNDARY)
