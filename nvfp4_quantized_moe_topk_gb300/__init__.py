"""GB300-native NVFP4 MoE expert layer (sm_103a CUDA kernels behind a C ABI).

The compute lives in ``libmoe_nvfp4.so`` (built from ``csrc/``); ``api`` is a
thin ctypes binding with the same entry-point names.  ``workload`` draws the
seeded synthetic inputs.  Importing this package does not load the CUDA
library; the first call into ``api`` does, and raises if it is missing.
"""
