"""fp64 CPU oracle of the paged-KV step -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library in ``paged_kv_cache_16_gb300``.
"""
