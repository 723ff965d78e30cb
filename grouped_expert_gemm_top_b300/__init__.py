"""B300-native (sm_103a) MoE expert layer: router, permute, grouped SwiGLU GEMMs,
combine and backward, exposed as a C-ABI library with a thin Python binding.

Submodules are imported on demand: ``inputs`` (seeded synthetic inputs, no
layer arithmetic), ``build`` (nvcc build of the shared library), ``moe``
(ctypes binding; raises if the CUDA library is missing).
"""
