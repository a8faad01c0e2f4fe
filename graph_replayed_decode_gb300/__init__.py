"""GB300-native fused serving step of a Qwen3/Qwen2.5-style dense decoder.

The compute path is the C-ABI library ``libeng.so`` (CUDA for sm_103a) declared in
``include/eng.h``; ``graph_replayed_decode_gb300.eng`` is its thin ctypes binding.
Importing this package does not load the library; the first binding call does,
and it raises if the library has not been built (there is no CPU fallback).
"""
