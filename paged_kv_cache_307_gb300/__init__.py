"""GB300-native paged KV-cache attention.

``libpa.so`` (built from ``csrc/`` by ``build.py``) holds the CUDA kernels
behind a C ABI declared in ``include/pa.h``; ``_lib`` is the thin ctypes
binding (argument marshalling only).  ``workloads`` draws the seeded
synthetic inputs.
"""

__all__ = ["build", "workloads"]
