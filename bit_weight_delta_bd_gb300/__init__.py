"""BitDelta multi-variant serving path for GB300 (sm_103a).

``bitdelta`` is the ctypes binding of libbitdelta.so (C ABI in
include/bitdelta.h); ``build`` compiles it; ``synth`` draws the seeded
synthetic inputs.  Importing the package loads nothing: the CUDA library is
opened on first use and its absence is an error, never a fallback.
"""
__all__ = ["bitdelta", "build", "synth"]
