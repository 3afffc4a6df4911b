"""GB300-native PRISM memory-recurrence forward (sm_103a).

The product is the C-ABI shared library built from ``csrc/`` (declared in
``include/prism.h``).  ``binding`` is a thin ctypes layer over it; it loads the
library on first use and raises if it is missing -- there is no CPU fallback.
"""
from .inputs import WORKLOADS, Workload, make_inputs, make_workload_inputs  # noqa: F401

__all__ = ["WORKLOADS", "Workload", "make_inputs", "make_workload_inputs"]
