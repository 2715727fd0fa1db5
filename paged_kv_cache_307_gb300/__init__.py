"""GB300-native paged KV-cache attention.

``libpa.so`` (built from ``csrc/`` by ``build.py``) holds the CUDA kernels
behind a C ABI declared in ``include/pa.h``; ``ops`` re-exports the thin
ctypes binding.  ``workloads`` draws the seeded synthetic inputs.
"""

__all__ = ["build", "workloads"]
