"""fp64 CPU oracle: test infrastructure, not part of the library.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA path never does. See
``oracle/attention.py`` for the definitions and the passages they follow.
"""
from .attention import *  # noqa: F401,F403
from .attention import __all__  # noqa: F401
