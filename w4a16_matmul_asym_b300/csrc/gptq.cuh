// gptq.cuh -- GPTQ quantization (second-order, column-greedy, with error feedback) into
// the asymmetric group-wise layout of w4_quantize_pack.
//
// Method ("Build a GPTQ INT4 Quantization Engine in Python/NumPy", Step 3): the columns
// of each row are quantized left to right; each column's quantization error, divided by
// U[j][j], is fed into the columns not yet quantized through row j of U, the upper
// Cholesky factor of H^-1.  Per row, values widened exactly to fp32, for j = 0 .. K-1:
//   at a group start (j % 128 == 0): s, zp of the current w[j .. j+127] by the rule of
//     w4_quantize_pack (fp32 min/max, s = (max - min) / 15 or 1, zp = clip(rint(-min /
//     s), 0, 15)); s16 = rne fp16(s);
//   q_j = clip(rint(w_j / s) + zp, 0, 15);
//   e   = (w_j - (q_j - zp) * s16) / U[j][j];
//   w_c = fma(-e, U[j][c], w_c) for c = j+1 .. K-1, in ascending j for every c.
// Every step is the IEEE fp32 operation (quotients by __fdiv_rn, fused multiply-adds),
// and each w_c receives its updates in ascending j, so the result is bit-exact with a
// sequential evaluation of the definition.
//
// Blocking without reordering.  The updates to a column can be deferred and applied
// later as long as each column still receives them in ascending j.  So the kernel walks
// 128-column blocks: (1) within the block, one warp per row runs the sequential sweep
// (lane l owns columns l + 32 i of the block in registers; every lane computes the
// current column's level and error from a shuffle of its value, so the warp never
// diverges), applying the in-block updates and recording the block's 128 errors;
// (2) then all threads apply those 128 errors, in order, to every later column of every
// row of the CTA: each thread owns one column for all rows, reads U[j][c] once per j
// (coalesced) and does one fused multiply-add per row.  The second phase is the O(N K^2)
// bulk of the work and runs at the CUDA cores' FMA rate; U (fp32 K x K) is read from L2
// once per CTA.
//
// Mapping: one CTA of 256 threads per band of R rows (R = 8 for K <= 4096, else 4); the
// band's working rows (R x K fp32), the block's diagonal part of U (128 x 128) and the
// errors (128 x R) live in shared memory.
#pragma once

#include "common.cuh"

namespace w4 {
namespace gptq {

constexpr int NUM_THREADS = 256;
constexpr int BLK = 128;                        // columns per block = group size
constexpr int SMEM_LIMIT = 227 * 1024;

__host__ __device__ constexpr int rows_for(int K) { return K <= 4096 ? 8 : 4; }
__host__ __device__ constexpr int smem_bytes(int K, int R) {
    return R * K * 4 + BLK * BLK * 4 + BLK * 8 * 4 + R * BLK;   // w, U block, errors, levels
}

struct Params {
    const void *W;        // fp16 or fp32 [N, K]
    const float *U;       // fp32 [K, K], upper triangular
    uint8_t *qweight;     // [N, K/2]
    __half *scales;       // [N, K/128]
    uint8_t *zeros;       // [N, K/128]
    int N, K, R;
};

template <bool kF32>
__global__ void __launch_bounds__(NUM_THREADS, 1) gptq_kernel(const Params p) {
    extern __shared__ __align__(16) float smem_f[];
    const int K = p.K, R = p.R;
    const int ng = K / BLK;
    float *w = smem_f;                               // [R][K]
    float *ub = w + R * K;                           // [128][128] diagonal block of U
    float *err = ub + BLK * BLK;                     // [128][8] errors of the block
    uint8_t *lev = reinterpret_cast<uint8_t *>(err + BLK * 8);   // [R][128] levels
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * R;
    const int rows = min(R, p.N - n0);

    // Working rows, widened exactly to fp32 (rows past N are zero and never stored);
    // 8 loads in flight per thread.
    for (int i0 = threadIdx.x; i0 < R * K; i0 += 8 * NUM_THREADS) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * NUM_THREADS;
            const int r = i / K, c = i - r * K;
            v[u] = 0.0f;
            if (i < R * K && r < rows) {
                const int64_t e = static_cast<int64_t>(n0 + r) * K + c;
                v[u] = kF32 ? __ldg(static_cast<const float *>(p.W) + e)
                            : __half2float(static_cast<const __half *>(p.W)[e]);
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (i0 + u * NUM_THREADS < R * K) w[i0 + u * NUM_THREADS] = v[u];
    }

    for (int b = 0; b < ng; ++b) {
        const int c0 = b * BLK;
        // The block's diagonal part of U: ub[jj][cc] = U[c0 + jj][c0 + cc].
        // (64 values per thread, 16 loads in flight.)
#pragma unroll 1
        for (int i0 = threadIdx.x; i0 < BLK * BLK; i0 += 16 * NUM_THREADS) {
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i = i0 + u * NUM_THREADS;
                v[u] = __ldg(p.U + static_cast<int64_t>(c0 + (i >> 7)) * K + c0 + (i & (BLK - 1)));
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) ub[i0 + u * NUM_THREADS] = v[u];
        }
        __syncthreads();

        // (1) the sequential sweep of the block, one warp per row.
        if (warp < R) {
            const int r = warp;
            float *wr = w + r * K + c0;
            float wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) wv[i] = wr[lane + 32 * i];
            // Group parameters from the current values (exact min/max, any order).
            float mn = fminf(fminf(wv[0], wv[1]), fminf(wv[2], wv[3]));
            float mx = fmaxf(fmaxf(wv[0], wv[1]), fmaxf(wv[2], wv[3]));
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
            const float s = (mx == mn) ? 1.0f : __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
            const float zp = fminf(fmaxf(rintf(__fdiv_rn(-mn, s)), 0.0f), 15.0f);
            const __half s16 = __float2half_rn(s);
            const float s16f = __half2float(s16);
            const float rs = __frcp_rn(s);
            if (lane == 0 && r < rows) {
                p.scales[static_cast<int64_t>(n0 + r) * ng + b] = s16;
                p.zeros[static_cast<int64_t>(n0 + r) * ng + b] = static_cast<uint8_t>(zp);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll 4
                for (int jl = 0; jl < 32; ++jl) {
                    const int jj = 32 * i + jl;
                    const float x = __shfl_sync(0xffffffffu, wv[i], jl);
                    // rint(x / s) from t = x * fl(1/s): within 2^-15 of a half-integer
                    // (or NaN) the IEEE quotient decides; beyond |t| > 32 both clip alike.
                    const float t = __fmul_rn(x, rs);
                    float rq = rintf(t);
                    if (!(fabsf(t - rq) <= 0.499969482421875f)) rq = rintf(__fdiv_rn(x, s));
                    const float q = fminf(fmaxf(__fadd_rn(rq, zp), 0.0f), 15.0f);
                    const float rec = __fmul_rn(__fsub_rn(q, zp), s16f);
                    const float e = __fdiv_rn(__fsub_rn(x, rec), ub[jj * BLK + jj]);
                    if (lane == jl) lev[r * BLK + jj] = static_cast<uint8_t>(q);
                    if (lane == 0) err[jj * 8 + r] = e;
#pragma unroll
                    for (int i2 = i; i2 < 4; ++i2) {
                        const int cc = lane + 32 * i2;
                        if (cc > jj) wv[i2] = __fmaf_rn(-e, ub[jj * BLK + cc], wv[i2]);
                    }
                }
            }
        }
        __syncthreads();

        // (2) the block's errors into every later column, in ascending j.
        const int rest = c0 + BLK;
        for (int c = rest + threadIdx.x; c < K; c += NUM_THREADS) {
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = r < R ? w[r * K + c] : 0.0f;
            const float *ucol = p.U + static_cast<int64_t>(c0) * K + c;
#pragma unroll 1
            for (int jb = 0; jb < BLK; jb += 32) {
                float uu[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) uu[k] = __ldg(ucol + static_cast<int64_t>(jb + k) * K);
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int jj = jb + k;
                    const float u = uu[k];
                    const float4 e0 = *reinterpret_cast<const float4 *>(err + jj * 8);
                    const float4 e1 = *reinterpret_cast<const float4 *>(err + jj * 8 + 4);
                    acc[0] = __fmaf_rn(-e0.x, u, acc[0]);
                    acc[1] = __fmaf_rn(-e0.y, u, acc[1]);
                    acc[2] = __fmaf_rn(-e0.z, u, acc[2]);
                    acc[3] = __fmaf_rn(-e0.w, u, acc[3]);
                    if (R > 4) {
                        acc[4] = __fmaf_rn(-e1.x, u, acc[4]);
                        acc[5] = __fmaf_rn(-e1.y, u, acc[5]);
                        acc[6] = __fmaf_rn(-e1.z, u, acc[6]);
                        acc[7] = __fmaf_rn(-e1.w, u, acc[7]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < R) w[r * K + c] = acc[r];
        }
        // The block's levels, packed: 64 bytes per row.
        for (int i = threadIdx.x; i < R * (BLK / 2); i += NUM_THREADS) {
            const int r = i >> 6, jb = i & 63;
            if (r < rows)
                p.qweight[static_cast<int64_t>(n0 + r) * (K / 2) + c0 / 2 + jb] =
                    static_cast<uint8_t>(lev[r * BLK + 2 * jb] | (lev[r * BLK + 2 * jb + 1] << 4));
        }
        __syncthreads();
    }
}

}  // namespace gptq
}  // namespace w4
