"""fp64 CPU oracle of the dropless MoE block -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU baseline / reference
leg of ``bench.py`` may import this package.  It shares no code with the CUDA
library and never imports it.
"""

from .dmoe_oracle import *  # noqa: F401,F403
from .dmoe_oracle import BLOCK  # noqa: F401
