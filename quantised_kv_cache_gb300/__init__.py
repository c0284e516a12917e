"""GB300-native TurboQuant-style KV-cache compression and compressed-cache decode attention.

The compute path is libtq.so (hand-written sm_103a CUDA behind a C ABI,
``include/tq.h``); ``tq`` is its ctypes binding and ``workloads`` draws the
seeded synthetic inputs. Importing the package does not load the library;
the first call into ``tq`` does, and fails loudly if it was never built.
"""

__all__ = ["tq", "workloads", "build"]
