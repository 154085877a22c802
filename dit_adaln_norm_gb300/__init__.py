"""GB300-native fused adaLN norm+modulate row kernels (sm_103a).

The kernels live in ``libdan.so`` (CUDA C++, C ABI, declared in
``include/dan.h``); ``dit_adaln_norm_gb300.ops`` is the thin ctypes binding
with the same entry-point names.  Importing the package loads nothing; the
first call into ``ops`` loads the library and raises if it is missing.
"""
__all__ = ["ops", "synth"]
