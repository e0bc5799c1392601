"""GB300 (sm_103a) paged mixed-codec decode attention.

The compute path is the C-ABI shared library ``libargus.so`` built from
``csrc/`` (see ``include/argus.h``); ``argus`` is its thin ctypes binding.
Importing this package does not load the library; ``argus.lib()`` does, and
raises if the library has not been built.
"""

__all__ = ["argus", "workloads"]
