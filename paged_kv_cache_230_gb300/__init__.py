"""GB300-native paged KV-cache decode attention.

The CUDA kernels and their C ABI live in ``csrc/`` (built into
``_lib/libpagedattn.so``); ``pagedattn`` is the thin ctypes binding;
``workloads`` draws seeded synthetic inputs.  Submodules are imported on
demand so that importing the input generator does not load the CUDA library.
"""
__all__ = ["pagedattn", "workloads", "build"]
