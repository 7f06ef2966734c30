"""GB300-native lossless cross-iteration exponent reuse for sharded bf16 weights.

The compute path is libciera (``include/ciera.h``): hand-written sm_103a
kernels behind a C ABI.  ``ciera`` is its thin Python binding,
``allgather.SimulatedAllgather`` drives one plan's device state, and
``workloads`` makes the seeded synthetic inputs.  Importing the package does
not load the CUDA library; the first call does, and fails loudly if it cannot.
"""
__all__ = ["ciera", "allgather", "workloads"]
