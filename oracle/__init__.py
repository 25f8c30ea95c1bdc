"""CPU oracle (test infrastructure only): see oracle.py and w4a16_oracle.c."""
from .oracle import (CALIB_METHODS, GROUP, REL_TOL, bf16_bits_to_f64, bf16_to_f64, build, check_y,
                     dequantize, dequantize16, f16_to_f32, f32_to_bf16_bits, f32_to_f16_bits,
                     gptq_factor, gptq_quantize, matmul, matmul_entries, mse_step, percentile_abs, quantize_pack,
                     quantize_act_int8, quantize_pack_calibrated, ulp_bf16, unpack, w4a8_matmul, w4a8_matmul_entries,
                     y_tolerance)

__all__ = ["CALIB_METHODS", "GROUP", "REL_TOL", "bf16_bits_to_f64", "bf16_to_f64", "build", "check_y",
           "dequantize", "dequantize16", "f16_to_f32", "f32_to_bf16_bits", "f32_to_f16_bits",
           "gptq_factor", "gptq_quantize", "matmul", "matmul_entries", "mse_step", "percentile_abs", "quantize_pack",
           "quantize_act_int8", "quantize_pack_calibrated", "ulp_bf16", "unpack", "w4a8_matmul", "w4a8_matmul_entries",
           "y_tolerance"]
