"""GB300 (sm_103a) implementation of the Quant VideoGen KV-cache compression path.

- ``video_kv_cache_gb300.qvg``   ctypes binding of the C ABI in include/qvg.h (libqvg.so)
- ``video_kv_cache_gb300.api``   allocation helpers over that binding (torch CUDA tensors)
- ``video_kv_cache_gb300.synth`` seeded synthetic video-shaped KV inputs and workloads
- ``video_kv_cache_gb300.build`` compiles libqvg.so for sm_103a

Nothing is loaded at import time; the first call into ``qvg`` loads libqvg.so and raises if
it is missing.
"""

__all__ = ["qvg", "api", "synth", "build"]
