"""CPU oracle for dynamic sparse prefill attention (test infrastructure only).

This package is a plain, slow, fp64 numpy restatement of what the CUDA path
computes.  It exists to check that path: only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product path never calls it, and it shares no code, table or helper with
the CUDA kernels.

Every function is pinned by ``tests/test_oracle_*.py`` against something other
than itself: library routines (torch scaled-dot-product attention in fp64,
``numpy.trace``), closed forms on margin-planted inputs, hand-worked masks in
``tests/golden/`` and invariants (probability mass, causality).  No function
here is "parity unpinned".
"""
from .mi_oracle import *  # noqa: F401,F403
from .mi_oracle import __all__ as _mi_all
from .mm_oracle import *  # noqa: F401,F403
from .mm_oracle import __all__ as _mm_all

__all__ = list(_mi_all) + list(_mm_all)
