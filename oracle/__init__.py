"""Independent double-precision CPU oracle (test infrastructure only).

Imported by the tests, by ``__graft_entry__.smoke()`` and by the CPU-baseline
and reference arms of ``bench.py``; never by the library itself."""
from .lopt_oracle import *  # noqa: F401,F403
