"""GB300-native speculative verify / accept / rollback for GatedDeltaNet (GDN) layers.

The compute path is libgdnspec.so (hand-written sm_103a CUDA kernels behind a C ABI,
include/gdnspec.h); ``speculative_verify_gdn_gb300._lib`` is its ctypes binding and
``speculative_verify_gdn_gb300.round`` runs one speculative round (verify -> accept -> rollback)
on preallocated device buffers. Importing the package loads nothing; the library is opened at the
first call and a missing build raises.
"""
__all__ = ["build", "inputs"]
