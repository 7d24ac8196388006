"""fp64 CPU oracle for row-wise LayerNorm / RMSNorm (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The CUDA library never does.
"""

from .norm_oracle import *  # noqa: F401,F403
from .norm_oracle import __all__  # noqa: F401
