// quantize_calib.cuh -- clip-range calibrated symmetric INT4 quantization + packing.
//
// Method ("Building a From-Scratch Group-Wise INT4 Quantization Layer for LLaMA
// Weights", Step 4, ScaleCalibrator), per group of 128 elements along K, values
// widened exactly to fp32:
//   percentile: r = the p-th percentile of |w|, linear interpolation between the
//     ascending order statistics a_0 <= ... <= a_127 in fp32: h = fl(fl(p / 100) * 127),
//     lo = floor(h), f = h - lo, r = a_lo + f * (a_(lo+1) - a_lo); step s = r / 7
//     (1 when r == 0).
//   mse: the step is searched over n candidates c_i = linspace(min|w|, max|w|, n)
//     (c_i = fl(min + fl(i * fl((max - min) / (n - 1)))), the last one max itself, the
//     only one min when n == 1); candidates below 1e-10 are skipped; each scores
//     fl(e / 128) with e the fp32 sum, in index order, of fl(d * d), d = fl(fl(t * c) - w),
//     t = clamp(rint(w / c), -7, 7); the first candidate with the smallest score wins
//     (1e-8 if none is scored).
//   Both: level = clamp(rint(w / s), -7, 7) + 8, zero point 8, scale = rne fp16(s), the
//   layout of w4_quantize_pack, so w4_matmul and w4_dequantize consume the result.
// Every step is an IEEE fp32 operation with round-to-nearest-even (the quotients by
// __fdiv_rn, the roundings to integers by rint), in the order above, so the result is
// bit-exact with a sequential fp32 evaluation.
//
// Mapping: one warp per group, lane l holding elements 4l .. 4l+3; a grid-stride loop
// over the flat group index G (W elements [128 G, 128 G + 128), qweight bytes
// [64 G, 64 G + 64), scales[G], zeros[G]).
//   percentile: the two order statistics it needs are found by repeated warp max- (or
//     min-) extraction when they lie within 8 of the top (or bottom) -- the usual
//     p = 99.9 takes two rounds -- and otherwise by a bitonic sort of the 128 magnitudes
//     (registers and xor-shuffles).  Either way the values are exact order statistics.
//   mse: the group goes to shared memory; lane l scores candidates l, l + 32, ... over
//     all 128 elements (broadcast reads), keeping its first minimum; a warp reduction
//     takes the smallest score, ties to the lower candidate index.  This is ALU work:
//     n * 128 quotients per group, each rounded from a reciprocal product except near a
//     tie (where the IEEE quotient is computed), which gives the same integer.
#pragma once

#include <climits>

#include "common.cuh"

namespace w4 {
namespace calib {

constexpr int WARPS = 8;
constexpr int NUM_THREADS = WARPS * 32;

struct Params {
    const void *W;        // fp16 or fp32 [N, K]
    int64_t groups;       // N * K / 128
    uint8_t *qweight;     // [N, K/2]
    __half *scales;       // [N, K/128]
    uint8_t *zeros;       // [N, K/128]
    float p;              // percentile, 0 < p <= 100
    int n;                // MSE candidates, >= 1
};

template <bool kF32>
__device__ __forceinline__ void load_group4(const void *W, int64_t g, int lane, float (&w)[4]) {
    if constexpr (kF32) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(W) + g * 32 + lane);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(W) + g * 32 + lane);
        w[0] = __half2float(__ushort_as_half(static_cast<unsigned short>(v.x & 0xFFFFu)));
        w[1] = __half2float(__ushort_as_half(static_cast<unsigned short>(v.x >> 16)));
        w[2] = __half2float(__ushort_as_half(static_cast<unsigned short>(v.y & 0xFFFFu)));
        w[3] = __half2float(__ushort_as_half(static_cast<unsigned short>(v.y >> 16)));
    }
}

// clamp(rint(w / s), -7, 7) + 8
__device__ __forceinline__ uint32_t level7(float w, float s) {
    const float t = fminf(fmaxf(rintf(__fdiv_rn(w, s)), -7.0f), 7.0f);
    return static_cast<uint32_t>(static_cast<int>(t) + 8);
}

// Levels of the lane's 4 elements -> 2 packed bytes; lane 0 also writes scale and zp.
__device__ __forceinline__ void store_group(const Params &p, int64_t g, int lane, const float (&w)[4], float s) {
    const uint32_t v = level7(w[0], s) | (level7(w[1], s) << 4) | (level7(w[2], s) << 8) | (level7(w[3], s) << 12);
    reinterpret_cast<uint16_t *>(p.qweight + g * 64)[lane] = static_cast<uint16_t>(v);
    if (lane == 0) {
        p.scales[g] = __float2half_rn(s);
        p.zeros[g] = 8;
    }
}

// Ascending bitonic sort of the warp's 128 values (element e = 4 lane + i in a[i]).
__device__ __forceinline__ void bitonic128(float (&a)[4], int lane) {
#pragma unroll
    for (int k = 2; k <= 128; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 4) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = lane * 4 + i;
                    const float o = __shfl_xor_sync(0xffffffffu, a[i], j >> 2);
                    const bool up = (e & k) == 0;
                    const bool lower = (e & j) == 0;
                    a[i] = (lower == up) ? fminf(a[i], o) : fmaxf(a[i], o);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if ((i & j) == 0) {
                        const bool up = ((lane * 4 + i) & k) == 0;
                        const float x = a[i], y = a[i | j];
                        a[i] = up ? fminf(x, y) : fmaxf(x, y);
                        a[i | j] = up ? fmaxf(x, y) : fminf(x, y);
                    }
                }
            }
        }
    }
}

// Element e of the sorted warp array (e uniform across the warp).
__device__ __forceinline__ float sorted_at(const float (&a)[4], int e) {
    const int i = e & 3;
    const float v = i == 0 ? a[0] : i == 1 ? a[1] : i == 2 ? a[2] : a[3];
    return __shfl_sync(0xffffffffu, v, e >> 2);
}

// The largest (kMax) or smallest remaining value of the warp's 128, returned to every
// lane, and one instance of it removed (the lowest lane, then the lowest register, that
// holds it; removed values become a sentinel outside [0, inf)).  Magnitudes only.
template <bool kMax>
__device__ __forceinline__ float extract(float (&a)[4], int lane) {
    const float sentinel = kMax ? -1.0f : __int_as_float(0x7f800000);
    float m = kMax ? fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])) : fminf(fminf(a[0], a[1]), fminf(a[2], a[3]));
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float t = __shfl_xor_sync(0xffffffffu, m, o);
        m = kMax ? fmaxf(m, t) : fminf(m, t);
    }
    const bool has = (a[0] == m) | (a[1] == m) | (a[2] == m) | (a[3] == m);
    const int owner = __ffs(__ballot_sync(0xffffffffu, has)) - 1;
    if (lane == owner) {
        if (a[0] == m) a[0] = sentinel;
        else if (a[1] == m) a[1] = sentinel;
        else if (a[2] == m) a[2] = sentinel;
        else a[3] = sentinel;
    }
    return m;
}

template <bool kF32>
__global__ void __launch_bounds__(NUM_THREADS) calib_percentile_kernel(const Params p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float qf = __fdiv_rn(p.p, 100.0f);
    const float h = __fmul_rn(qf, 127.0f);
    const float fl = floorf(h);
    const int lo = min(max(static_cast<int>(fl), 0), 127);
    const int hi = min(lo + 1, 127);
    const float f = __fsub_rn(h, fl);
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * WARPS + warp; g < p.groups;
         g += static_cast<int64_t>(gridDim.x) * WARPS) {
        float w[4], a[4];
        load_group4<kF32>(p.W, g, lane, w);
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = fabsf(w[i]);
        float alo, ahi;
        if (lo >= 120) {                      // from the top: round r gives a_(127 - r)
            alo = ahi = 0.0f;
            for (int r = 0; r <= 127 - lo; ++r) {
                const float v = extract<true>(a, lane);
                if (r == 127 - hi) ahi = v;
                if (r == 127 - lo) alo = v;
            }
        } else if (hi <= 7) {                 // from the bottom: round r gives a_r
            alo = ahi = 0.0f;
            for (int r = 0; r <= hi; ++r) {
                const float v = extract<false>(a, lane);
                if (r == lo) alo = v;
                if (r == hi) ahi = v;
            }
        } else {
            bitonic128(a, lane);
            alo = sorted_at(a, lo);
            ahi = sorted_at(a, hi);
        }
        const float r = __fadd_rn(alo, __fmul_rn(f, __fsub_rn(ahi, alo)));
        const float s = (r == 0.0f) ? 1.0f : __fdiv_rn(r, 7.0f);
        store_group(p, g, lane, w, s);
    }
}

// Percentiles near either end of the group (lo >= 120, or hi <= 7): one thread per
// group.  The thread keeps the KT largest (or smallest) magnitudes of its 128 in a
// sorted register list (each value bubbles through the list: one max and one min per
// slot), so the two order statistics come without warp exchanges; the levels use
// t = w * fl(1/s), which gives clamp(rint(w / s), -7, 7) exactly except within 2^-15 of
// a half-integer (|t - fl(w/s)| <= 8 * 3 * 2^-24 there; beyond |t| > 8 both clamp),
// where the IEEE quotient is taken.
template <bool kF32, bool kTop, int KT>
__global__ void __launch_bounds__(NUM_THREADS) calib_percentile_ends_kernel(const Params p) {
    const float qf = __fdiv_rn(p.p, 100.0f);
    const float h = __fmul_rn(qf, 127.0f);
    const float fl = floorf(h);
    const int lo = min(max(static_cast<int>(fl), 0), 127);
    const int hi = min(lo + 1, 127);
    const float f = __fsub_rn(h, fl);
    // Positions in the kept list: from the top, a_(127 - r) is entry r; from the bottom, a_r.
    const int rlo = kTop ? 127 - lo : lo, rhi = kTop ? 127 - hi : hi;
    constexpr int VPL = kF32 ? 4 : 8;          // values per 16-byte load
    constexpr int LOADS = 128 / VPL;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * NUM_THREADS + threadIdx.x; g < p.groups;
         g += static_cast<int64_t>(gridDim.x) * NUM_THREADS) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.W) + g * LOADS;
        float keep[KT];
#pragma unroll
        for (int j = 0; j < KT; ++j) keep[j] = kTop ? -1.0f : __int_as_float(0x7f800000);
#pragma unroll 4
        for (int l = 0; l < LOADS; ++l) {
            const uint4 v = __ldg(src + l);
            float x[VPL];
            if constexpr (kF32) {
                x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
                x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
            } else {
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    x[2 * k] = __half2float(__ushort_as_half(static_cast<unsigned short>(u[k] & 0xFFFFu)));
                    x[2 * k + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(u[k] >> 16)));
                }
            }
#pragma unroll
            for (int e = 0; e < VPL; ++e) {
                float c = fabsf(x[e]);
                if (!(c == c)) c = kTop ? -1.0f : __int_as_float(0x7f800000);   // NaN: left out
#pragma unroll
                for (int j = 0; j < KT; ++j) {
                    const float a = kTop ? fmaxf(keep[j], c) : fminf(keep[j], c);
                    c = kTop ? fminf(keep[j], c) : fmaxf(keep[j], c);
                    keep[j] = a;
                }
            }
        }
        float alo = keep[0], ahi = keep[0];
#pragma unroll
        for (int j = 1; j < KT; ++j) {
            if (j == rlo) alo = keep[j];
            if (j == rhi) ahi = keep[j];
        }
        const float r = __fadd_rn(alo, __fmul_rn(f, __fsub_rn(ahi, alo)));
        const float sc = (r == 0.0f) ? 1.0f : __fdiv_rn(r, 7.0f);
        const float rs = __frcp_rn(sc);
        // Levels: the group again (L1/L2), 8 levels -> one 32-bit word.
        uint32_t *dst = reinterpret_cast<uint32_t *>(p.qweight + g * 64);
        uint32_t prev = 0;
#pragma unroll 2
        for (int l = 0; l < LOADS; ++l) {
            const uint4 v = __ldg(src + l);
            float x[VPL];
            if constexpr (kF32) {
                x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
                x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
            } else {
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    x[2 * k] = __half2float(__ushort_as_half(static_cast<unsigned short>(u[k] & 0xFFFFu)));
                    x[2 * k + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(u[k] >> 16)));
                }
            }
            uint32_t word = 0;
#pragma unroll
            for (int e = 0; e < VPL; ++e) {
                const float t = __fmul_rn(x[e], rs);
                float q = rintf(t);
                if (!(fabsf(t - q) <= 0.499969482421875f)) q = rintf(__fdiv_rn(x[e], sc));
                q = fminf(fmaxf(q, -7.0f), 7.0f);
                word |= static_cast<uint32_t>(static_cast<int>(q) + 8) << (4 * ((l * VPL + e) & 7));
            }
            if constexpr (kF32) {
                // 4 levels per load: two loads make one word
                if (l & 1) dst[l >> 1] = prev | word;
                else prev = word;
            } else {
                dst[l] = word;
            }
        }
        p.scales[g] = __float2half_rn(sc);
        p.zeros[g] = 8;
    }
}

__device__ __forceinline__ float candidate(int i, int n, float lo, float hi, float step) {
    if (n == 1) return lo;
    if (i == n - 1) return hi;
    return __fadd_rn(lo, __fmul_rn(static_cast<float>(i), step));
}

template <bool kF32>
__global__ void __launch_bounds__(NUM_THREADS) calib_mse_kernel(const Params p) {
    __shared__ __align__(16) float sw[WARPS][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float4 *sw4 = reinterpret_cast<const float4 *>(sw[warp]);
    const int n = p.n;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * WARPS + warp; g < p.groups;
         g += static_cast<int64_t>(gridDim.x) * WARPS) {
        float w[4];
        load_group4<kF32>(p.W, g, lane, w);
        reinterpret_cast<float4 *>(sw[warp])[lane] = make_float4(w[0], w[1], w[2], w[3]);
        float lo = fminf(fminf(fabsf(w[0]), fabsf(w[1])), fminf(fabsf(w[2]), fabsf(w[3])));
        float hi = fmaxf(fmaxf(fabsf(w[0]), fabsf(w[1])), fmaxf(fabsf(w[2]), fabsf(w[3])));
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        __syncwarp();
        const float step = n > 1 ? __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(n - 1)) : 0.0f;
        float best = __int_as_float(0x7f800000);   // +inf
        int bi = INT_MAX;
        for (int i = lane; i < n; i += 32) {
            const float c = candidate(i, n, lo, hi, step);
            if (c < 1e-10f) continue;
            const float rc = __frcp_rn(c);          // finite: c >= 1e-10
            float e = 0.0f;
#pragma unroll 4
            for (int k4 = 0; k4 < 32; ++k4) {
                const float4 v = sw4[k4];
                const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    // rint of the IEEE quotient: from x * fl(1/c) (within 3 ulp of it)
                    // unless that lies within 2^-16 of a half-integer (or is not
                    // finite), where the quotient itself is taken.  Beyond |x| = 7.5 the
                    // clamp makes both give +-7.
                    const float xr = __fmul_rn(x[u], rc);
                    float r = rintf(xr);
                    if (!(fabsf(__fsub_rn(xr, r)) < 0.4999847412109375f)) r = rintf(__fdiv_rn(x[u], c));
                    const float t = fminf(fmaxf(r, -7.0f), 7.0f);
                    const float d = __fsub_rn(__fmul_rn(t, c), x[u]);
                    e = __fadd_rn(e, __fmul_rn(d, d));
                }
            }
            const float mse = __fdiv_rn(e, 128.0f);
            if (mse < best) {
                best = mse;
                bi = i;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ob < best || (ob == best && oi < bi)) {
                best = ob;
                bi = oi;
            }
        }
        const float s = (bi == INT_MAX) ? 1e-8f : candidate(bi, n, lo, hi, step);
        store_group(p, g, lane, w, s);
        __syncwarp();
    }
}

}  // namespace calib
}  // namespace w4
