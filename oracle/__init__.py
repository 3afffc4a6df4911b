"""fp64 CPU oracle for the PRISM memory-recurrence forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA library.
"""
from .prism_oracle import build, forward  # noqa: F401
