"""GB300-native decode attention over a sub-byte quantized paged KV cache.

The compute lives in libkvq.so (CUDA kernels for sm_103a behind the C ABI of include/kvq.h);
``quantized_paged_kv_int4_gb300.kvq`` is its Python binding, ``workloads`` the seeded synthetic
inputs used by the tests and the benchmark.
"""
