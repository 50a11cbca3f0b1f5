"""GB300 (sm_103a) W4A16 routed-MoE decode block: CUDA kernels behind a C ABI, with a thin ctypes binding.

Importing the package is cheap; the shared library is loaded on first use by ``w4a16_top_mixture_gb300.lib``
and a missing or unloadable library raises instead of falling back to anything else.
"""
