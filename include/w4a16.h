/*
 * w4a16.h -- C ABI of the B300 (sm_103a) library for group-wise asymmetric INT4
 * weight-only quantization and the fused dequantize-matmul (W4A16) that consumes it.
 *
 * Data convention (all tensors dense, row-major, resident in device memory):
 *   W        fp16 or fp32  [N, K]      weights, N = out_features, K = in_features
 *   qweight  uint8         [N, K/2]    4-bit levels q, two per byte: element 2j of a
 *                                      row in the low nibble, element 2j+1 in the high
 *   scales   fp16          [N, K/128]  per-group scale, rounded to nearest-even fp16
 *   zeros    uint8         [N, K/128]  per-group zero point, 0..15, one per byte
 *   A        bf16          [M, K]      activations
 *   Y        bf16          [M, N]      output, Y = A * W_hat^T, fp32 accumulation,
 *                                      rounded to nearest-even bf16
 * Groups are 128 contiguous elements along K of one row of W.
 *
 * Ownership: the caller allocates and owns every buffer; the library allocates no
 * device or host memory, keeps no per-call state, and holds no pointer after return.
 * Asynchrony: every call enqueues work on the caller's stream and returns without
 * synchronizing.  On a validation failure a call returns before launching anything
 * and leaves every output untouched.
 * Thread safety: calls may be made from any host thread; the only process-wide
 * state is a cache of per-device attributes and the test hooks at the end.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define W4_API __attribute__((visibility("default")))
#else
#define W4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    W4_OK = 0,
    W4_ERR_INVALID_ARG = 1,   /* negative size, null pointer for a non-empty tensor,
                                 K not a multiple of the group, unknown dtype */
    W4_ERR_UNSUPPORTED = 2,   /* valid but not implemented: group size other than 128 */
    W4_ERR_MISALIGNED = 3,    /* a pointer violates the alignment stated below */
    W4_ERR_CUDA = 4,          /* a CUDA runtime/driver call or a launch failed */
    W4_ERR_TIMEOUT = 5        /* a kernel gave up a bounded wait (see w4_check_device_error) */
} w4_status;

/* Element types: of W for w4_quantize_pack / w4_quantize_pack_sym (F16, F32), of the
 * output of w4_dequantize (F16, BF16). */
typedef enum { W4_DTYPE_F16 = 0, W4_DTYPE_F32 = 1, W4_DTYPE_BF16 = 2 } w4_dtype;

#define W4_GROUP_SIZE 128

/*
 * w4_quantize_pack -- quantize W[N,K] to 4-bit levels with one fp16 scale and one
 * uint8 zero point per group of 128 elements along K, and pack the levels.
 *
 * Defined by: "From-Scratch INT4 Weight-Only Quantizer with Per-Group Scales and
 * Zero-Points" (Architecture Overview, item 3; Steps 5-6: per-group min/max, scale =
 * (max-min)/15, zero point = round(-min/scale) clipped to [0,15]); "From Scratch:
 * Building a GPTQ INT4 Quantizer in Pure Python" (Step 2: q = clip(round(w/scale +
 * zero_point), 0, 15)); "Build a GPTQ INT4 Quantization Engine in Python/NumPy"
 * (Step 4: two levels per byte, element 2j in the low nibble).  Exact convention:
 * per group, with values widened exactly to fp32,
 *     s  = (max == min) ? 1 : (max - min) / 15              (fp32, IEEE division)
 *     zp = clip(round_half_even(-min / s), 0, 15)
 *     q  = clip(round_half_even(w / s) + zp, 0, 15)         (IEEE fp32 division by s)
 *     scales = fp16_round_nearest_even(s), zeros = zp.
 * Results are bit-exact with that definition for finite inputs whose per-group range
 * max-min is finite in fp32 (always true for fp16 input).
 *
 * Arguments:
 *   W        device pointer, fp16 or fp32 [N, K] per w_dtype; 16-byte aligned.
 *   w_dtype  W4_DTYPE_F16 or W4_DTYPE_F32.
 *   N, K     rows and columns; N >= 0, K >= 0, K % group == 0.
 *   group    must be 128 (other positive values: W4_ERR_UNSUPPORTED).
 *   qweight  device pointer, uint8 [N, K/2]; 16-byte aligned.  Written.
 *   scales   device pointer, fp16 [N, K/128]; 2-byte aligned.  Written.
 *   zeros    device pointer, uint8 [N, K/128].  Written.
 *   stream   the stream to run on (0 = legacy default stream).
 * N == 0 or K == 0 is an empty problem: returns W4_OK and launches nothing.
 */
W4_API int w4_quantize_pack(const void *W, int w_dtype, int64_t N, int64_t K, int group,
                     uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream);

/*
 * w4_quantize_pack_sym -- the symmetric variant of w4_quantize_pack: per group of 128
 * elements along K, with values widened exactly to fp32,
 *     s  = (absmax == 0) ? 1 : absmax / 7                 (fp32, IEEE division;
 *                                                           absmax = max |w| of the group)
 *     q  = clip(round_half_even(w / s), -8, 7)            (IEEE fp32 division by s)
 *     scales = fp16_round_nearest_even(s), zeros = 8, stored level = q + 8,
 * i.e. the layout of w4_quantize_pack with every zero point 8, so that w4_matmul and
 * w4_dequantize consume it unchanged ((level - 8) * s = q * s).  Since |w / s| <= 7 up
 * to the rounding of the quotient, the stored levels lie in [1, 15].
 *
 * Defined by: "Build a GPTQ INT4 Quantization Engine in Python/NumPy" (Step 2: per-group
 * absmax, scale = absmax / 7 with 1 for an all-zero group, q = clip(round(w / scale),
 * -8, 7)); "Building a From-Scratch Group-Wise INT4 Quantization Layer for LLaMA
 * Weights" (Key design decisions: symmetric per-group scales as the standard choice for
 * transformer weights).  Bit-exact with the definition above for finite inputs.
 *
 * Arguments, alignment, empty problems and errors: as w4_quantize_pack.
 */
W4_API int w4_quantize_pack_sym(const void *W, int w_dtype, int64_t N, int64_t K, int group,
                                uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream);

/*
 * w4_dequantize -- materialize W_hat[N,K] = (q - zp) * scale_fp16 as a 16-bit tensor,
 * the explicit dequantize path for a consumer that wants the whole weight matrix.
 *
 * Defined by: "From Scratch: Building a GPTQ INT4 Quantizer in Pure Python" (Step 4:
 * dequantize = (q - zero_point) * scale).  Exact convention: the product (q - zp) * s16
 * is exact in fp32 and is rounded once to nearest-even bf16 (out_dtype W4_DTYPE_BF16)
 * or fp16 (W4_DTYPE_F16; a magnitude past the fp16 range gives +-inf).  Bit-exact.
 *
 * Arguments:
 *   qweight, scales, zeros  as written by w4_quantize_pack or w4_quantize_pack_sym
 *            (same alignment rules).
 *   N, K     N >= 0, K >= 0, K % group == 0.
 *   group    must be 128.
 *   out_dtype W4_DTYPE_BF16 or W4_DTYPE_F16 (others: W4_ERR_INVALID_ARG).
 *   out      device pointer, 16-bit [N, K]; 16-byte aligned.  Written.
 *   stream   the stream to run on.
 * N == 0 or K == 0: W4_OK, nothing launched.
 */
W4_API int w4_dequantize(const uint8_t *qweight, const void *scales, const uint8_t *zeros, int64_t N,
                         int64_t K, int group, int out_dtype, void *out, cudaStream_t stream);

/*
 * w4_matmul -- Y[M,N] = A[M,K] * W_hat[N,K]^T with W_hat = (q - zp) * scale_fp16,
 * dequantized on the fly (the full-precision W is never materialized), fp32
 * accumulation, output rounded to nearest-even bf16.
 *
 * Defined by: "From Scratch: Building a GPTQ INT4 Quantizer in Pure Python" (Step 4:
 * dequantize = (q - zero_point) * scale); "Build a GPTQ INT4 Quantization Engine in
 * Python/NumPy" (Step 5: the fused dequantize-matmul y = x W^T over packed weights);
 * "Building a From-Scratch Group-Wise INT4 Quantization Layer for LLaMA Weights"
 * (Architecture Overview and Step 2: dequantization fused with the matmul as the hot
 * path).  Accuracy contract, per output element:
 *     |Y - Y_exact| <= 8e-3 * sum_k |A[m,k] * W_hat[n,k]| + ulp_bf16(|Y_exact|) / 2.
 * Paths: M = 1 runs integer dot products (dp4a) on exact block-floating-point
 * activation digits; 2 <= M <= 8 a CUDA-core split-K GEMV (bf16 x bf16 -> fp32 FMA);
 * 9 <= M <= 16 with fewer 128-row tiles than three quarters of the SMs a tcgen05 kernel
 * that splits K across tensor-memory lanes; otherwise a tcgen05 tensor-core GEMM
 * (bf16 x bf16 -> fp32 in tensor memory) on weight tiles dequantized into tensor memory.
 * Shapes a fast path cannot take (K not a multiple of 2048, unaligned scale or zero
 * tables) run a plain CUDA-core kernel.
 *
 * Arguments:
 *   A        device pointer, bf16 [M, K]; 16-byte aligned.
 *   M, N, K  M >= 0, N >= 0, K >= 0, K % group == 0.
 *   group    must be 128.
 *   qweight, scales, zeros  as written by w4_quantize_pack (same alignment rules).
 *   Y        device pointer, bf16 [M, N]; 2-byte aligned.  Written.
 *   stream   the stream to run on.
 * M == 0 or N == 0: W4_OK, nothing launched.  K == 0: Y is filled with zeros.
 */
W4_API int w4_matmul(const void *A, int64_t M, int64_t N, int64_t K, int group,
              const uint8_t *qweight, const void *scales, const uint8_t *zeros,
              void *Y, cudaStream_t stream);

/* A static, human-readable name for a status code (never NULL). */
W4_API const char *w4_status_string(int status);

/*
 * w4_check_device_error -- synchronize `stream`, then read and clear the library's
 * device error word for the current device.  Kernels never trap: every wait on a
 * barrier or copy is bounded, and a wait that runs out records W4_ERR_TIMEOUT in the
 * error word and lets the kernel exit cleanly (in-flight copies drained, tensor
 * memory freed).  Returns W4_OK, W4_ERR_TIMEOUT, or W4_ERR_CUDA if the
 * synchronization itself failed.
 */
W4_API int w4_check_device_error(cudaStream_t stream);

/*
 * Test hooks (process-wide, for the failure-detection tests; not for production use).
 *   w4_set_wait_timeout_ns: limit of every bounded wait in nanoseconds of
 *     %globaltimer (default 2e9, i.e. two seconds; 0 restores the default).
 *   w4_debug_inject_stall: when nonzero, the next kernel launches make their
 *     consumer wait on a barrier that nothing ever signals, so the bounded wait must
 *     run out, record W4_ERR_TIMEOUT and exit; the setting stays until cleared.
 */
W4_API void w4_set_wait_timeout_ns(uint64_t ns);
W4_API void w4_debug_inject_stall(int enable);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
