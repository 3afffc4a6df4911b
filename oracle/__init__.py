"""fp64 CPU oracles for the PRISM memory-recurrence forward, its backward pass (prism_backward)
and the block's input projections (prism_projection) -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA library.
"""
from .prism_oracle import build, forward  # noqa: F401
