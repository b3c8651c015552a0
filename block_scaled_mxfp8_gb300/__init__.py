"""MXFP8 block-scaled attention (forward + backward) for NVIDIA GB300 (sm_103a).

The compute path is libmxa.so (CUDA C++, tcgen05 / TMEM / TMA), declared in
include/mxa.h; ``block_scaled_mxfp8_gb300.mxa`` is its ctypes binding and
``block_scaled_mxfp8_gb300.build`` compiles it in-tree.  ``inputs`` holds the
seeded synthetic workloads.
"""
__all__ = ["mxa", "build", "inputs"]
