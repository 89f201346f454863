"""fp64 CPU oracle: test infrastructure, not part of the library.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA path never does. See
``oracle/attention.py`` (attention over a paged cache, prefill, merges) and
``oracle/flat_gemm.py`` (the decode-phase flat GEMM) for the definitions and the
passages they follow.
"""
from .attention import *  # noqa: F401,F403
from .attention import __all__ as _attention_all
from .flat_gemm import *  # noqa: F401,F403
from .flat_gemm import __all__ as _flat_gemm_all

__all__ = list(_attention_all) + list(_flat_gemm_all)
