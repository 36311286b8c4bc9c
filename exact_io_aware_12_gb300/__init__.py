"""Exact IO-aware attention for GB300 (sm_103a).

The compute lives in a C-ABI shared library of hand-written CUDA kernels
(``csrc/``, declared in ``include/fa.h``).  This package holds the build step,
a thin ctypes binding with the same names as the C entry points, and the
seeded workload generator.  Importing the package does not load the library;
the first call does, and fails loudly if the library is missing.
"""
from .workloads import WORKLOADS, Workload  # noqa: F401

__all__ = ["WORKLOADS", "Workload"]
