"""GB300-native KV4-RL decode hot path: paged INT4 KV cache with a bounded INT8 side cache.

The compute path is libkv4 (CUDA, sm_103a) behind the C ABI in include/kv4.h;
``kv4`` is its Python binding (argument marshalling only).
"""
