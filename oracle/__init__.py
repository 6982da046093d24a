"""CPU oracle for LazyAttention's hot path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product path never imports, calls or links it.  Parity status of
every function is recorded in ``lazy_oracle``'s module docstring: all are pinned; none is
"parity unpinned".
"""
from .lazy_oracle import *  # noqa: F401,F403
from . import lazy_oracle  # noqa: F401
