"""CPU fp64 oracle for exact tiled attention (test infrastructure only).

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py``; the CUDA library never uses it.
"""
from .attention import *  # noqa: F401,F403
from .attention import __all__  # noqa: F401
