"""GB300-native group-quantised KV-cache attention (sm_103a).

The compute path is the C-ABI library ``libkvq.so`` (CUDA kernels for
sm_103a); :mod:`attention_group_quantized_gb300.kvq` is its thin Python
binding.  Importing this package does not load the library; the binding
loads it on first use and raises if it is missing.
"""
__all__ = ["kvq"]
