"""CPU oracle for the DSA lightning-indexer step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.
"""

from .dsa_oracle import *  # noqa: F401,F403
from .sparse_mla import *  # noqa: F401,F403
