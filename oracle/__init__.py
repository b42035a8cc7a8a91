"""CPU oracle (test infrastructure only; see ``oracle/cp_oracle.py``).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The product path never does.
"""
from .cp_oracle import *  # noqa: F401,F403
from .cp_oracle import MASK_MIN  # noqa: F401
