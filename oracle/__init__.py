"""fp64 CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

``attention`` is the plain numpy definition; ``c_oracle`` is the same
definition in C (OpenMP over rows) used for timed CPU baselines; ``plan_rule``
restates the split-KV plan rule in pure Python; ``kv_append`` writes new
tokens' K/V rows into a paged cache (E4M3 quantisation for fp8 pools);
``mla`` is multi-latent attention decode over a paged latent cache.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use
this package; the product path never imports it.
"""
