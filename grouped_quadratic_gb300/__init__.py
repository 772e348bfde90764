"""GB300-native OAL grouped-quadratic causal attention.

The compute lives in the CUDA library ``liboal.so`` (sources under ``csrc/``,
C ABI declared in ``include/oal.h``); ``grouped_quadratic_gb300.oal`` is the
thin ctypes binding with the same entry-point names.  ``inputs`` holds the
seeded synthetic workloads.  Importing the package loads nothing; the binding
loads the library on first use and raises if it is missing.
"""
__all__ = ["oal", "inputs"]
