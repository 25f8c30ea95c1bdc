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
 * Ownership: the caller allocates and owns every buffer (including the scratch
 * workspace w4_matmul_w4a8 may ask for); the library allocates no device or host
 * memory, keeps no per-call state, and holds no pointer after return.  The one
 * exception is the fixed scratch array of w4_matmul_w4a8_noalloc: a static device array
 * of W4_NOALLOC_SCRATCH_BYTES in every GPU context that loads the library.
 * Asynchrony: every call enqueues work on the caller's stream and returns without
 * synchronizing.  On a validation failure a call returns before launching anything
 * and leaves every output untouched.
 * Thread safety: calls may be made from any host thread; the only process-wide
 * state is a cache of per-device attributes (including the device address of that
 * scratch array) and the test hooks at the end.
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
    W4_ERR_TIMEOUT = 5,       /* a kernel gave up a bounded wait (see w4_check_device_error) */
    W4_ERR_SCRATCH_LIMIT = 6  /* w4_matmul_w4a8_noalloc: the shape needs more scratch than
                                 W4_NOALLOC_SCRATCH_BYTES */
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
 * w4_quantize_pack_percentile / w4_quantize_pack_mse -- symmetric quantization with a
 * calibrated clip range per group of 128 elements along K, in the layout of
 * w4_quantize_pack (every zero point 8), so that w4_matmul and w4_dequantize consume
 * the result unchanged.
 *
 * Defined by: "Building a From-Scratch Group-Wise INT4 Quantization Layer for LLaMA
 * Weights" (Step 4, ScaleCalibrator: the percentile of |w| as the clip range, and the
 * search over linspace(min|w|, max|w|, n) candidate steps minimizing the reconstruction
 * MSE with levels round(w / s).clamp(-7, 7)).  Exact convention, per group, values
 * widened exactly to fp32, every operation IEEE fp32 with round-to-nearest-even:
 *   percentile (0 < p <= 100): sort |w| ascending (a_0 .. a_127); h = (p / 100) * 127,
 *     lo = floor(h), f = h - lo, r = a_lo + f * (a_min(lo+1,127) - a_lo);
 *     s = (r == 0) ? 1 : r / 7.
 *   mse (candidates = n >= 1): c_i = min|w| + i * ((max|w| - min|w|) / (n - 1)) for
 *     i < n - 1, c_(n-1) = max|w| (n == 1: c_0 = min|w|); skip c_i < 1e-10; score(c) =
 *     (sum over k = 0..127 in order of d_k * d_k) / 128 with d_k = clamp(rint(w_k / c),
 *     -7, 7) * c - w_k; s = the first c_i with the smallest score (1e-8 if none).
 *   level = clamp(round_half_even(w / s), -7, 7) + 8, zeros = 8,
 *   scales = fp16_round_nearest_even(s).
 * Bit-exact with that definition for finite inputs (for mse: |w| small enough that the
 * squared errors stay finite in fp32, e.g. any fp16 input).  The mse search performs
 * n * 128 divisions per group: an offline calibration step, bound by arithmetic.
 *
 * Arguments, alignment, empty problems and errors: as w4_quantize_pack; p outside
 * (0, 100] or candidates outside [1, 2^24] give W4_ERR_INVALID_ARG.
 */
W4_API int w4_quantize_pack_percentile(const void *W, int w_dtype, int64_t N, int64_t K, int group,
                                       float p, uint8_t *qweight, void *scales, uint8_t *zeros,
                                       cudaStream_t stream);
W4_API int w4_quantize_pack_mse(const void *W, int w_dtype, int64_t N, int64_t K, int group,
                                int candidates, uint8_t *qweight, void *scales, uint8_t *zeros,
                                cudaStream_t stream);

/*
 * w4_matmul_w4a8_noalloc -- w4_matmul_w4a8 for callers that cannot allocate device
 * memory: the same computation, arguments and results, but the scratch that
 * w4_matmul_w4a8 takes from the caller (on shapes outside the decode path) comes from a
 * fixed array inside the library, W4_NOALLOC_SCRATCH_BYTES (16 MiB) on every GPU that
 * loads the library, held until the process exits.  The sources have no counterpart of
 * this call; it exists for the library's users.
 *
 * Who needs it: callers that cannot or must not allocate device memory at the point of
 * the call: plugins and extensions whose host framework owns all device memory through
 * its own pool and gives them no way into it; real-time inference loops that must not
 * allocate after start-up, because an allocation can synchronize the device and stall
 * the loop; code paths with no way to recover from an allocation failure.
 *
 * Allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * Limit: shapes whose scratch (w4_matmul_w4a8_workspace_size(M, K), i.e. M * K * 2
 *   bytes off the decode path) exceeds W4_NOALLOC_SCRATCH_BYTES return
 *   W4_ERR_SCRATCH_LIMIT before anything is launched; decode shapes need none.
 * First call on a device: looks up the array's device address (cudaGetSymbolAddress,
 *   once per device, with that device current) and caches it.  Make that first call on
 *   each device before any stream capture begins.
 * Sharing: every call on a device uses the same array, and it keeps what the last call
 *   left there.  Nothing in it needs to start at zero: each call writes the part it
 *   reads (the widened activations) before reading it.  Calls whose work overlaps on the
 *   GPU (on different streams, or from different host threads without ordering) race on
 *   the array and corrupt each other's results; order them on one stream or with events.
 * Errors: as w4_matmul_w4a8, plus W4_ERR_SCRATCH_LIMIT.
 */
#define W4_NOALLOC_SCRATCH_BYTES (16u << 20)
W4_API int w4_matmul_w4a8_noalloc(const int8_t *a_q, const float *a_scale, int64_t M, int64_t N, int64_t K,
                                  int group, const uint8_t *qweight, const void *scales,
                                  const uint8_t *zeros, void *Y, cudaStream_t stream);

/*
 * w4_gptq_quantize -- GPTQ: quantize W[N,K] into the layout of w4_quantize_pack (4-bit
 * levels, fp16 scales, uint8 zero points per group of 128 along K), column by column,
 * feeding each column's quantization error into the columns not yet quantized.
 *
 * Defined by: "Build a GPTQ INT4 Quantization Engine in Python/NumPy" (Step 3: the
 * Hessian of the calibration activations, the Cholesky factor of its inverse, and the
 * column-greedy quantization with error propagation).  Exact convention, per row, values
 * widened exactly to fp32, every step an IEEE fp32 operation (fused multiply-add for
 * the updates):
 *   for j = 0 .. K-1:
 *     if j % 128 == 0: s, zp of the current w[j .. j+127] by the rule of
 *       w4_quantize_pack; scales = s16 = fp16_round_nearest_even(s), zeros = zp;
 *     q_j = clip(round_half_even(w_j / s) + zp, 0, 15);
 *     e   = (w_j - (q_j - zp) * s16) / U[j][j];
 *     w_c = fma(-e, U[j][c], w_c) for every c > j (each w_c updated in ascending j).
 * Bit-exact with that definition.  U is the caller's: the upper-triangular Cholesky
 * factor of H^-1 (H^-1 = U^T U, H the damped Hessian X^T X / n + damp I of the
 * calibration activations X), fp32 [K, K] row-major; only its upper triangle is read
 * and its diagonal must be nonzero.
 *
 * Arguments:
 *   W        device pointer, fp16 or fp32 [N, K] per w_dtype; 16-byte aligned.
 *   N, K     N >= 0, K >= 0, K % group == 0; K <= 8192 (W4_ERR_UNSUPPORTED above).
 *   group    must be 128.
 *   U        device pointer, fp32 [K, K]; 16-byte aligned.
 *   qweight, scales, zeros  outputs as in w4_quantize_pack.
 *   stream   the stream to run on.
 * N == 0 or K == 0: W4_OK, nothing launched.  The work is O(N K^2) fused multiply-adds
 * (an offline step, bound by the FMA rate).
 */
W4_API int w4_gptq_quantize(const void *W, int w_dtype, int64_t N, int64_t K, int group, const float *U,
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
 * activation digits; 2 <= M <= 16 warp-level tensor-core MMAs (bf16 x bf16 -> fp32)
 * on weights dequantized in registers, when K is a multiple of 2048, the scale and zero
 * tables are 16-byte aligned and the activations fit in shared memory; M >= 9 otherwise
 * a tcgen05 tensor-core GEMM (bf16 x bf16 -> fp32 in tensor memory) on weight tiles
 * dequantized into tensor memory.  M <= 8 shapes those paths cannot take (K not a
 * multiple of 2048, unaligned tables, activations too large) run a CUDA-core GEMV.
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

/*
 * w4_quantize_act_int8 -- per-token INT8 dynamic quantization of the activations (the
 * A8 of W4A8).
 *
 * Defined by: "Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization with
 * Per-Channel Scale" (Step 3, activations_to_int8: per token, scale = max|A| / 127 with
 * max|A| clipped below at 1e-8, levels round(A / scale) clipped to [-128, 127]).  Exact
 * convention, per row m of A, values widened exactly to fp32:
 *     a_scale[m] = max(max_k |A[m,k]|, 1e-8) / 127          (IEEE fp32 division)
 *     a_q[m,k]   = clip(round_half_even(A[m,k] / a_scale[m]), -128, 127)
 * Bit-exact for finite A (|a_q| <= 127 then).
 *
 * Arguments:
 *   A        device pointer, bf16 [M, K]; 16-byte aligned.
 *   M, K     M >= 0, K >= 0, K % 8 == 0.
 *   a_q      device pointer, int8 [M, K]; 16-byte aligned.  Written.
 *   a_scale  device pointer, fp32 [M]; 4-byte aligned.  Written.
 *   stream   the stream to run on.
 * M == 0: W4_OK, nothing launched.
 */
W4_API int w4_quantize_act_int8(const void *A, int64_t M, int64_t K, int8_t *a_q, float *a_scale,
                                cudaStream_t stream);

/*
 * w4_matmul_w4a8 -- Y[M,N] = a_scale[m] * sum_k a_q[m,k] * W_hat[n,k] with W_hat =
 * (q - zp) * scale_fp16, fp32 accumulation, output rounded to nearest-even bf16: the
 * W4A8 forward pass over per-token INT8 activations.
 *
 * Defined by: "Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization with
 * Per-Channel Scale" (Step 5, forward_quant: the INT8 activations times their per-token
 * scale, multiplied by the dequantized INT4 weights).  Accuracy contract per element:
 *     |Y - Y_exact| <= 8e-3 * sum_k |a_q[m,k] a_scale[m] W_hat[n,k]| + ulp_bf16(|Y_exact|) / 2.
 * Paths, none of them using the int8 tensor pipe (this part's int8 tensor rate is far
 * below its bf16 rate):
 *   M = 1, K a multiple of 2048 up to 16384: integer dot products (dp4a) of the int8
 *     activations with the 4-bit levels, exact in int32 per group; no workspace.
 *   1 <= M <= 16 otherwise, K a multiple of 2048 (activations fitting in shared memory):
 *     the decode kernel of w4_matmul, a_q widened to bf16 while staged (int8 x int4
 *     products are exact in bf16 x bf16 -> fp32); no workspace.
 *   otherwise: a_q is widened to bf16 into `workspace` and the tcgen05 GEMM of w4_matmul
 *     runs with a_scale applied to each output row before rounding.
 *
 * Arguments:
 *   a_q, a_scale  as written by w4_quantize_act_int8 (a_q 16-byte aligned).
 *   M, N, K, group, qweight, scales, zeros, Y  as w4_matmul; on the decode path scales
 *            and zeros must be 16-byte aligned (W4_ERR_MISALIGNED otherwise).
 *   workspace  device pointer to at least w4_matmul_w4a8_workspace_size(M, K) bytes,
 *            16-byte aligned, owned by the caller; may be NULL when that size is 0.
 *            A smaller workspace gives W4_ERR_INVALID_ARG.  Its contents are scratch.
 *   stream   the stream to run on.
 * M == 0 or N == 0: W4_OK, nothing launched.  K == 0: Y is filled with zeros.
 */
W4_API size_t w4_matmul_w4a8_workspace_size(int64_t M, int64_t K);
W4_API int w4_matmul_w4a8(const int8_t *a_q, const float *a_scale, int64_t M, int64_t N, int64_t K,
                          int group, const uint8_t *qweight, const void *scales, const uint8_t *zeros,
                          void *Y, void *workspace, size_t workspace_bytes, cudaStream_t stream);

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
