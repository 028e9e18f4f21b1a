"""TurboQuant / PolarQuant KV-cache compression and attention over the
compressed cache, for NVIDIA GB300 (sm_103a).

The compute lives in libtq.so (C ABI, include/tq.h); ``binding`` is the thin
ctypes layer over it.  Import ``turboquant_kv_cache_gb300.binding`` for the
calls; ``inputs`` holds the seeded synthetic workloads."""

__all__ = ["binding", "inputs"]
