"""B300-native decode-step KV page retrieval and sparse GQA attention.

The CUDA library (``libkvr.so``) and its ctypes binding live in
``kv_cache_page_build_b300.kvr``; the seeded workload generator in
``kv_cache_page_build_b300.synth``.  Importing the package loads neither.
"""
