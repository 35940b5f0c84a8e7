"""Float64 CPU oracle of the DFlash draft-attention step (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The library never imports it.
"""
from . import dflash_oracle  # noqa: F401
