"""GB300-native Palu G-LRD decode attention over a latent KV cache.

``rank_kv_cache_gb300.palu`` is the Python binding of the C ABI in
``include/palu_attn.h`` (it loads ``_lib/libpalu_attn.so`` and fails loudly if
the library has not been built); ``rank_kv_cache_gb300.build`` compiles it.
"""
