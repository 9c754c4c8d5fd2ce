"""CPU oracle for KIVI grouped asymmetric KV-cache quantization.

TEST INFRASTRUCTURE ONLY.  A plain C restatement of the method (kivi_ref.c),
loaded through ctypes by the tests, the smoke check and the benchmark's CPU
baseline.  The CUDA library (``kivi_bit_kv_gb300``) never imports this package
and this package never imports the library.
"""
