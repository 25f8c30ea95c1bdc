"""B300-native group-wise asymmetric INT4 weight-only quantization and W4A16 matmul.

The compute lives in libw4a16.so (hand-written CUDA for sm_103a behind a C ABI,
declared in include/w4a16.h).  This package is its thin Python binding.
"""
from ._binding import (EXPORTED, GROUP_SIZE, LIB_PATH, W4_DTYPE_BF16, W4_DTYPE_F16, W4_DTYPE_F32,
                       W4_ERR_CUDA, W4_ERR_INVALID_ARG, W4_ERR_MISALIGNED, W4_ERR_SCRATCH_LIMIT, W4_ERR_TIMEOUT,
                       W4_NOALLOC_SCRATCH_BYTES,
                       W4_ERR_UNSUPPORTED, W4_OK, W4Error, dequantize, gptq_quantize, load_library, matmul,
                       matmul_w4a8, quantize_act_int8, quantize_pack, status_string,
                       w4_check_device_error, w4_matmul_w4a8, w4_matmul_w4a8_noalloc,
                       w4_matmul_w4a8_workspace_size,
                       w4_gptq_quantize, w4_quantize_act_int8,
                       w4_debug_inject_stall, w4_dequantize, w4_matmul, w4_quantize_pack,
                       w4_quantize_pack_mse, w4_quantize_pack_percentile, w4_quantize_pack_sym,
                       w4_set_wait_timeout_ns)

__all__ = ["EXPORTED", "GROUP_SIZE", "LIB_PATH", "W4_DTYPE_BF16", "W4_DTYPE_F16", "W4_DTYPE_F32",
           "W4_ERR_CUDA", "W4_ERR_INVALID_ARG", "W4_ERR_MISALIGNED", "W4_ERR_SCRATCH_LIMIT", "W4_ERR_TIMEOUT",
           "W4_NOALLOC_SCRATCH_BYTES",
           "W4_ERR_UNSUPPORTED", "W4_OK", "W4Error", "dequantize", "gptq_quantize", "load_library", "matmul",
           "matmul_w4a8", "quantize_act_int8", "quantize_pack", "status_string", "w4_check_device_error",
           "w4_debug_inject_stall", "w4_gptq_quantize", "w4_matmul_w4a8", "w4_matmul_w4a8_noalloc", "w4_matmul_w4a8_workspace_size", "w4_quantize_act_int8",
           "w4_dequantize", "w4_matmul", "w4_quantize_pack", "w4_quantize_pack_mse",
           "w4_quantize_pack_percentile", "w4_quantize_pack_sym", "w4_set_wait_timeout_ns"]
