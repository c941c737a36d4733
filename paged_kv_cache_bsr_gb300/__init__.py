"""GB300 (sm_103a) attention over a block-sparse (paged) KV cache.

The compute lives in libpkvbsr.so (C ABI: include/pkv_bsr.h); ``api`` is its
thin ctypes binding, ``runner`` marshals workloads through it, ``workloads``
draws seeded synthetic inputs, and ``build`` compiles the library.
"""
__version__ = "0.1.0"

__all__ = ["api", "build", "runner", "workloads"]
