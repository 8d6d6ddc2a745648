"""Fused linear cross-entropy for GB300 (sm_103a).

The compute path is the C-ABI library ``libflce.so`` (hand-written CUDA);
``binding`` is its thin ctypes wrapper.  Importing this package does not load
the library; ``binding.lib()`` does, and fails loudly if it was not built.
"""
__all__ = ["inputs", "binding"]
