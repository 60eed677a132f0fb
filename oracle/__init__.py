"""fp64 CPU oracle for exact tiled attention — TEST INFRASTRUCTURE ONLY.

Only tests/, the package smoke check and the benchmark's CPU-baseline leg
import this package. The CUDA library never does, and shares no code with it.

  ref.py     the plain definition: fp64 attention forward and backward
  online.py  the online-softmax recurrence, tile by tile (for the pages'
             worked examples and as a cross-check of ref.py)
  arith.py   the size / traffic / work arithmetic the pages print

Parity status: every function is pinned (tests/test_oracle.py) except the
"FlashAttention" page's 4.19 GiB tiled-traffic figure, which no reading of
the text reproduces; no function computes it, so nothing depends on it.
"""
from . import arith, online, ref  # noqa: F401
