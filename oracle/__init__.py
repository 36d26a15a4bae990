"""CPU oracle for layer-end KV-cache compression (test infrastructure only).

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg.  It shares no code with the CUDA library.
"""

from . import kvc_oracle  # noqa: F401
from .kvc_oracle import *  # noqa: F401,F403
