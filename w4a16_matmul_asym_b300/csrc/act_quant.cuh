// act_quant.cuh -- per-token INT8 dynamic activation quantization (the A8 of W4A8) and
// the exact int8 -> bf16 expansion the tensor-core GEMM consumes.
//
// Method ("Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization with
// Per-Channel Scale", Step 3, activations_to_int8), per token = row m of A[M,K], the
// bf16 values widened exactly to fp32:
//   s_a[m]    = max(max_k |A[m,k]|, 1e-8) / 127             (IEEE fp32 division)
//   a_q[m,k]  = clip(round_half_even(A[m,k] / s_a[m]), -128, 127)   (IEEE quotient)
// Bit-exact with that sequential fp32 definition: the maximum is exact in any order and
// every quotient is the correctly rounded __fdiv_rn.
//
// Mapping: one warp per row (grid-stride over rows).  Pass 1 reads the row in 16-byte
// pieces (8 bf16) and reduces |a| to the row maximum (lane maxima, then xor-shuffles);
// pass 2 reads the row again (from L2: a row is at most a few tens of KB) and writes 8
// int8 levels per piece as one 8-byte store.  Memory-bound at 3 bytes per element.
#pragma once

#include "common.cuh"

namespace w4 {
namespace actq {

constexpr int WARPS = 8;
constexpr int NUM_THREADS = WARPS * 32;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t level8(float a, float s) {
    const float t = fminf(fmaxf(rintf(__fdiv_rn(a, s)), -128.0f), 127.0f);
    return static_cast<uint32_t>(static_cast<int>(t)) & 0xFFu;
}

// K a multiple of 8; A 16-byte aligned rows (K * 2 bytes apart), a_q 8-byte aligned rows.
__global__ void __launch_bounds__(NUM_THREADS)
    act_quant_int8_kernel(const __nv_bfloat16 *__restrict__ A, int64_t M, int64_t K, int8_t *__restrict__ a_q,
                          float *__restrict__ a_scale) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t pieces = K >> 3;
    for (int64_t m = static_cast<int64_t>(blockIdx.x) * WARPS + warp; m < M;
         m += static_cast<int64_t>(gridDim.x) * WARPS) {
        const uint4 *row = reinterpret_cast<const uint4 *>(A + m * K);
        float amax = 0.0f;
        for (int64_t i = lane; i < pieces; i += 32) {
            const uint4 v = __ldg(row + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = __fdiv_rn(fmaxf(amax, 1e-8f), 127.0f);
        uint2 *out = reinterpret_cast<uint2 *>(a_q + m * K);
        for (int64_t i = lane; i < pieces; i += 32) {
            const uint4 v = __ldg(row + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t b[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                b[2 * j] = level8(bf16_lo(w[j]), s);
                b[2 * j + 1] = level8(bf16_hi(w[j]), s);
            }
            out[i] = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                                b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
        }
        if (lane == 0) a_scale[m] = s;
    }
}

// int8 [n] -> bf16 [n] (exact: |x| <= 128 needs 8 significant bits), 8 per thread-step.
__global__ void __launch_bounds__(256)
    int8_to_bf16_kernel(const int8_t *__restrict__ src, __nv_bfloat16 *__restrict__ dst, int64_t n8) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(src) + i);
        const uint32_t w[2] = {v.x, v.y};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float lo = static_cast<float>(static_cast<int8_t>((w[h] >> (16 * j)) & 0xFFu));
                const float hi = static_cast<float>(static_cast<int8_t>((w[h] >> (16 * j + 8)) & 0xFFu));
                const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
                o[2 * h + j] = *reinterpret_cast<const uint32_t *>(&b);
            }
        }
        reinterpret_cast<uint4 *>(dst)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace actq
}  // namespace w4
