"""GB300-native fused grouped-query attention forward.

The compute lives in a C-ABI shared library built from ``csrc/`` for sm_103a;
``binding`` marshals arguments to it.  Importing this package does not load
the library; the first call does, and it raises if the library is missing.
"""
from . import workloads  # noqa: F401  (seeded synthetic inputs; no attention arithmetic)

__all__ = ["workloads"]
