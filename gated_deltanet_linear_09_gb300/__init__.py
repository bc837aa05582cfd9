"""GB300-native Gated DeltaNet (gated delta rule) layer library.

The compute lives in libgdn.so (CUDA for sm_103a, C ABI in include/gdn.h).  ``gdn`` is the
ctypes binding with the same entry-point names, ``runtime`` a small device-memory helper
around it, ``synth`` the seeded synthetic-input generator.  Submodules are imported on
demand so that building or generating inputs does not need a GPU.
"""
__all__ = ["gdn", "runtime", "synth", "build"]
