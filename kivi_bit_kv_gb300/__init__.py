"""kivi_bit_kv_gb300 -- KIVI grouped asymmetric KV-cache quantization on GB300.

The compute path is libkivi.so (include/kivi.h), hand-written CUDA for sm_103a:
prefix encode of keys (per channel) and values (per token), materialize,
token append with group flush, and decode attention with dequantization fused
into the loads.  This package is its thin Python binding; torch provides
device memory and streams.

    from kivi_bit_kv_gb300 import KiviCache, abi
    cache = KiviCache(B, H, D, bits_k=2, bits_v=2, G=32, R=128, Tmax=...)
    abi.kivi_quant_keys(cache, K); abi.kivi_quant_values(cache, V)
"""
from . import abi
from .abi import KiviError
from .cache import KiviCache

__all__ = ["abi", "KiviCache", "KiviError"]
