"""DeepSeekMoE layer forward for one B300 (sm_103a).

The compute lives in libmoe.so (C ABI in include/moe.h; CUDA kernels under
csrc/).  ``moe`` is its ctypes binding, ``layer`` a small holder of device
buffers built on it, ``inputs`` the seeded synthetic workloads.  Submodules
are imported on demand so that ``inputs`` can be used without the library.
"""
__all__ = ["moe", "layer", "inputs", "build"]
