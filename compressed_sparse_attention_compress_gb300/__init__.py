"""GB300-native compressed sparse attention forward (DeepSeek-V4 CSA / HCA / window-only).

The compute path is the C-ABI library ``libcsa.so`` built from ``csrc/`` for
sm_103a; ``api`` is a thin ctypes binding over it.  Importing this package does
not load the library: ``api`` does, and fails loudly when it is missing.
"""
__all__ = ["inputs", "workload"]
