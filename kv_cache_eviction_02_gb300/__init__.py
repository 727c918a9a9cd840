"""GB300-native KV-cache eviction pass (LORE-KV projected deletion scores, H2O decode eviction).

The compute runs in the CUDA library ``libkvevict.so`` behind the C-ABI declared in
``include/kvevict.h``; :mod:`kv_cache_eviction_02_gb300.api` is the thin binding.
"""
