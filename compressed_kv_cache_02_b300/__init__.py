"""TurboQuant hot path on B300: rotate + scalar-code + QJL-sign quantization and
the asymmetric estimator behind a C-ABI library (``libtq.so``) of sm_103a kernels.

``compressed_kv_cache_02_b300.tq`` is the thin ctypes binding; importing it loads
the library and fails loudly when it is missing.  ``inputs`` draws seeded synthetic data.
"""
