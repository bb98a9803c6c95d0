"""MAC-Attention per-step decode attention for GB300 (sm_103a).

The compute path is ``libmac_gb300.so`` (hand-written CUDA kernels behind a
C ABI, declared in ``include/mac.h``); ``mac`` is its thin ctypes binding.
Import ``long_context_decode_gb300.mac`` to load the library: it raises if the
library has not been built, there is no fallback.
"""
__all__ = ["mac", "workloads"]
