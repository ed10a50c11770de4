"""Test infrastructure: the float64 CPU oracle for FAVOR+ forward attention.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.
"""
from .favor64 import *  # noqa: F401,F403
from .favor64 import __all__  # noqa: F401
