"""GB300-native block-quantized weight rows (Q4_0 / Q8_0).

The compute path is the CUDA library libbq.so (C ABI, see include/bq.h); the
Python binding in .binding only marshals device pointers and sizes to it.
"""
from .binding import (  # noqa: F401
    Q4_0, Q8_0, Q4_1, Q5_0, Q5_1, Q4_K, Q6_K, BQError, block_values, block_bytes, quantize_rows, dequantize_rows, gemv, gemv_multi, gemv_sequence, attn_decode, gemm,
    kv_quantize, kv_write, kv_bias, BASIS_PLAIN, BASIS_HADAMARD64, block_dots, lib, library_path,
)
