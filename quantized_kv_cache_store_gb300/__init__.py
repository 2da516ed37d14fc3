"""TurboQuant speculative-verify decode attention over a quantised paged KV
cache, hand-written CUDA for sm_103a behind a small C ABI (libtqkv.so).

The binding in :mod:`quantized_kv_cache_store_gb300.tqkv` only marshals
arguments; every step of the path runs in the CUDA kernels.  There is no CPU
fallback: calling into the binding without the compiled library raises.
"""
