// act_quant.cuh -- per-token INT8 dynamic activation quantization (the A8 of W4A8) and
// the exact int8 -> bf16 expansion the tensor-core GEMM consumes.
//
// Method ("Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization with
// Per-Channel Scale", Step 3, activations_to_int8), per token = row m of A[M,K], the
// bf16 values widened exactly to fp32:
//   s_a[m]    = max(max_k |A[m,k]|, 1e-8) / 127             (IEEE fp32 division)
//   a_q[m,k]  = clip(round_half_even(A[m,k] / s_a[m]), -128, 127)   (IEEE quotient)
// Bit-exact with that sequential fp32 definition: the maximum is exact in any order and
// every level is the one the correctly rounded quotient gives (below).
//
// Mapping, few rows (decode): one CTA of 256 threads per row; each thread loads up to 8
// 16-byte pieces (8 bf16 each) of the row into registers and reduces |a| to its
// maximum, the row maximum goes through shared memory (no warp shuffles), and the
// levels are computed from the registers and stored as one 8-byte word per piece
// (rows up to 16384 elements are read once).  Many rows (prefill): a warp per row, two
// passes over the row (measured faster there than the CTA-per-row form).
//
// The CTA-per-row kernel avoids a division per element: t = a * fl(1/s) lies within
// |a/s| 3 2^-24 <= 2.3e-5 of the IEEE quotient fl(a/s) (|a/s| <= 127 + ulp), so
// whenever t is farther than 2^-15 from a half-integer, rint(t) == rint(fl(a/s)).
// Elements inside that window (and NaN) take the IEEE division __fdiv_rn.
#pragma once

#include "common.cuh"

namespace w4 {
namespace actq {

constexpr int NUM_THREADS = 256;
constexpr int REG_PIECES = 8;                 // 16-byte pieces per thread kept in registers
constexpr float kTieSlack = 0.499969482421875f;  // 0.5 - 2^-15

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// clip(rint(a / s), -128, 127) as a byte, with a / s the IEEE fp32 quotient.
__device__ __forceinline__ uint32_t level8(float a, float s, float rs) {
    const float t = __fmul_rn(a, rs);
    float r = rintf(t);
    if (!(fabsf(t - r) <= kTieSlack)) r = rintf(__fdiv_rn(a, s));
    const float c = fminf(fmaxf(r, -128.0f), 127.0f);
    return static_cast<uint32_t>(static_cast<int>(c)) & 0xFFu;
}
__device__ __forceinline__ float piece_absmax(const uint4 &v, float m) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    return m;
}
// The same level by the IEEE division alone (straight-line code, no per-element branch).
__device__ __forceinline__ uint32_t level8_div(float a, float s) {
    const float c = fminf(fmaxf(rintf(__fdiv_rn(a, s)), -128.0f), 127.0f);
    return static_cast<uint32_t>(static_cast<int>(c)) & 0xFFu;
}
template <bool kRcp>
__device__ __forceinline__ uint2 piece_levels(const uint4 &v, float s, float rs) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t b[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        b[2 * j] = kRcp ? level8(bf16_lo(w[j]), s, rs) : level8_div(bf16_lo(w[j]), s);
        b[2 * j + 1] = kRcp ? level8(bf16_hi(w[j]), s, rs) : level8_div(bf16_hi(w[j]), s);
    }
    return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// K a multiple of 8; A 16-byte aligned rows (K * 2 bytes apart), a_q 8-byte aligned rows.
// Few rows: one row per CTA of 256 threads, the row held in registers.
__global__ void __launch_bounds__(NUM_THREADS)
    act_quant_int8_kernel(const __nv_bfloat16 *__restrict__ A, int64_t M, int64_t K, int8_t *__restrict__ a_q,
                          float *__restrict__ a_scale) {
    __shared__ float wmax[NUM_THREADS / 32];
    __shared__ float tmax[NUM_THREADS];
    const int t = threadIdx.x;
    const int64_t pieces = K >> 3;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4 *row = reinterpret_cast<const uint4 *>(A + m * K);
        uint2 *out = reinterpret_cast<uint2 *>(a_q + m * K);
        uint4 v[REG_PIECES];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < REG_PIECES; ++j) {
            const int64_t i = t + static_cast<int64_t>(j) * NUM_THREADS;
            v[j] = i < pieces ? __ldg(row + i) : make_uint4(0, 0, 0, 0);
            amax = piece_absmax(v[j], amax);
        }
        for (int64_t i = t + static_cast<int64_t>(REG_PIECES) * NUM_THREADS; i < pieces; i += NUM_THREADS)
            amax = piece_absmax(__ldg(row + i), amax);
        // Row maximum: per thread -> per warp (its first thread) -> every thread.
        tmax[t] = amax;
        __syncthreads();
        if ((t & 31) == 0) {
            float wm = tmax[t];
#pragma unroll 8
            for (int k = 1; k < 32; ++k) wm = fmaxf(wm, tmax[t + k]);
            wmax[t >> 5] = wm;
        }
        __syncthreads();
        float rowmax = wmax[0];
#pragma unroll
        for (int k = 1; k < NUM_THREADS / 32; ++k) rowmax = fmaxf(rowmax, wmax[k]);
        const float s = __fdiv_rn(fmaxf(rowmax, 1e-8f), 127.0f);
        const float rs = __frcp_rn(s);
#pragma unroll
        for (int j = 0; j < REG_PIECES; ++j) {
            const int64_t i = t + static_cast<int64_t>(j) * NUM_THREADS;
            if (i < pieces) out[i] = piece_levels<true>(v[j], s, rs);
        }
        for (int64_t i = t + static_cast<int64_t>(REG_PIECES) * NUM_THREADS; i < pieces; i += NUM_THREADS)
            out[i] = piece_levels<true>(__ldg(row + i), s, rs);
        if (t == 0) a_scale[m] = s;
        __syncthreads();   // tmax / wmax are rewritten for the next row
    }
}

// Many rows: a warp per row (8 per CTA, grid-stride), two passes over the row (the
// maximum, then the levels by IEEE division; the second read comes from L2), the row
// maximum by xor shuffles once per row.
__global__ void __launch_bounds__(NUM_THREADS)
    act_quant_int8_rows_kernel(const __nv_bfloat16 *__restrict__ A, int64_t M, int64_t K,
                               int8_t *__restrict__ a_q, float *__restrict__ a_scale) {
    constexpr int WARPS = NUM_THREADS / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t pieces = K >> 3;
    for (int64_t m = static_cast<int64_t>(blockIdx.x) * WARPS + warp; m < M;
         m += static_cast<int64_t>(gridDim.x) * WARPS) {
        const uint4 *row = reinterpret_cast<const uint4 *>(A + m * K);
        float amax = 0.0f;
        for (int64_t i = lane; i < pieces; i += 32) amax = piece_absmax(__ldg(row + i), amax);
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = __fdiv_rn(fmaxf(amax, 1e-8f), 127.0f);
        uint2 *out = reinterpret_cast<uint2 *>(a_q + m * K);
        for (int64_t i = lane; i < pieces; i += 32) out[i] = piece_levels<false>(__ldg(row + i), s, 0.0f);
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
