// quantize_pack.cuh -- group-wise asymmetric INT4 quantization + nibble packing.
//
// Method ("From-Scratch INT4 Weight-Only Quantizer with Per-Group Scales and
// Zero-Points", Architecture Overview item 3 and Steps 5-6; "From Scratch: Building a
// GPTQ INT4 Quantizer in Pure Python", Step 2; packing per "Build a GPTQ INT4
// Quantization Engine in Python/NumPy", Step 4), per group of 128 along K:
//   s  = (max == min) ? 1 : (max - min) / 15          fp32, IEEE division
//   zp = clip(rhe(-min / s), 0, 15)
//   q  = clip(rhe(w / s) + zp, 0, 15)                 IEEE fp32 quotient
//   qweight byte j of a group = q[2j] | q[2j+1] << 4; scale stored as rne fp16(s).
//
// Layout: the flat group index G = n * (K/128) + g addresses every output directly:
// qweight bytes [64 G, 64 G + 64), scales[G], zeros[G], and W elements
// [128 G, 128 G + 128).  So the kernel walks groups as one flat array.
//
// Mapping: a half-warp owns a group; each lane holds 8 consecutive elements (one
// 16-byte load for fp16, two for fp32).  A warp iteration covers 8 groups (2 KB of
// fp16 W), with all four 512-byte warp loads issued before any is consumed.  Min and
// max come from an 8-element local pass plus a 4-step xor-shuffle across the half
// warp; each lane then writes its 8 nibbles as one 32-bit word, so a warp stores
// 128 contiguous bytes per pair of groups.
//
// Quotient w/s without a divide per element: t = w * fl(1/s) lies within 3 ulp of the
// IEEE quotient x = fl(w/s) (two roundings of 2^-24 relative each, plus x's own).
// For |t| <= 64 that is below 2^-16, so whenever t is farther than 2^-16 from a
// half-integer, rhe(t) == rhe(x).  Only elements inside that window (about 3e-5 of
// them) take the IEEE division __fdiv_rn.  Elements with |t| > 31.5 clip to level 0
// or 15 whichever integer they round to, so their rounding needs no care.
// Rounding to an integer uses the add-1.5*2^23 trick: for |t| < 2^22,
// fl(t + 1.5*2^23) = 1.5*2^23 + rhe(t) exactly; adding zp into the constant first is
// exact too, and outside ties rhe(t + zp) == rhe(t) + zp.  The level is then the low
// 4 bits of the clamped float's bit pattern.
#pragma once

#include "common.cuh"

namespace w4 {

constexpr float kRoundMagic = 12582912.0f;              // 1.5 * 2^23
constexpr uint32_t kRoundMagicBits = 0x4B400000u;       // bit pattern of kRoundMagic
constexpr float kHalfMinusSlack = 0.4999847412109375f;  // 0.5 - 2^-16

struct GroupParams {
    float s;       // fp32 scale
    float rcp;     // fl(1/s)
    float mz;      // kRoundMagic + zp (exact)
    float zp;      // zero point as float (0..15)
};

__device__ __forceinline__ GroupParams group_params(float mn, float mx) {
    GroupParams p;
    p.s = (mx == mn) ? 1.0f : __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    const float zq = rintf(__fdiv_rn(-mn, p.s));
    p.zp = fminf(fmaxf(zq, 0.0f), 15.0f);
    p.rcp = __frcp_rn(p.s);
    p.mz = __fadd_rn(kRoundMagic, p.zp);
    return p;
}

// Returns kRoundMagic + clip(rhe(w / s) + zp, 0, 15) as a float (bits 0x4B40000q).
__device__ __forceinline__ float quantize_one(float w, const GroupParams &p) {
    const float t = __fmul_rn(w, p.rcp);
    float v = __fadd_rn(t, p.mz);
    const float e = __fsub_rn(t, __fsub_rn(v, p.mz));
    if (fabsf(e) > kHalfMinusSlack) {
        // Near a half-integer: take the IEEE quotient and round it half-to-even.
        const float x = __fdiv_rn(w, p.s);
        const float k = __fsub_rn(__fadd_rn(x, kRoundMagic), kRoundMagic);  // rhe(x), |x| < 2^22
        v = (fabsf(x) < 4194304.0f) ? __fadd_rn(kRoundMagic, __fadd_rn(k, p.zp)) : __fadd_rn(x, p.mz);
    }
    return fminf(fmaxf(v, kRoundMagic), kRoundMagic + 15.0f);
}

// Packs 8 levels (each as the float kRoundMagic + q) into one 32-bit word, element i
// in bits [4i, 4i+4): sum_i (bits_i - magic) * 16^i, computed mod 2^32.
__device__ __forceinline__ uint32_t pack8(const float (&v)[8]) {
    uint32_t acc = 0u - kRoundMagicBits * 0x11111111u;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc += __float_as_uint(v[i]) * (1u << (4 * i));
    return acc;
}

template <bool kF32>
__global__ void __launch_bounds__(256) quantize_pack_kernel(const void *__restrict__ W,
                                                            int64_t total_groups,
                                                            uint32_t *__restrict__ qw,
                                                            __half *__restrict__ scales,
                                                            uint8_t *__restrict__ zeros) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;  // which group of a pair this lane works on
    const int sub = lane & 15;   // 8-element slice of the group
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

    for (int64_t base = warp * 8; base < total_groups; base += nwarps * 8) {
        uint4 raw[4][kF32 ? 2 : 1];
        // Issue all loads of the iteration first.
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t g = base + 2 * j + half;
            const int64_t e = g * 128 + sub * 8;
            if (g < total_groups) {
                if constexpr (kF32) {
                    const float *Wf = static_cast<const float *>(W);
                    raw[j][0] = ldg_stream_16(Wf + e);
                    raw[j][1] = ldg_stream_16(Wf + e + 4);
                } else {
                    raw[j][0] = ldg_stream_16(static_cast<const __half *>(W) + e);
                }
            } else {
#pragma unroll
                for (int u = 0; u < (kF32 ? 2 : 1); ++u) raw[j][u] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t g = base + 2 * j + half;
            float w[8];
            float mn, mx;
            if constexpr (kF32) {
                const float *f = reinterpret_cast<const float *>(&raw[j][0]);
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = f[i];
                mn = fminf(fminf(fminf(w[0], w[1]), fminf(w[2], w[3])),
                           fminf(fminf(w[4], w[5]), fminf(w[6], w[7])));
                mx = fmaxf(fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3])),
                           fmaxf(fmaxf(w[4], w[5]), fmaxf(w[6], w[7])));
            } else {
                const __half2 *h = reinterpret_cast<const __half2 *>(&raw[j][0]);
                // min/max on packed halves (exact), then widen the two survivors.
                const __half2 lo = __hmin2(__hmin2(h[0], h[1]), __hmin2(h[2], h[3]));
                const __half2 hi = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
                mn = fminf(__low2float(lo), __high2float(lo));
                mx = fmaxf(__low2float(hi), __high2float(hi));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __half22float2(h[i]);
                    w[2 * i] = f.x;
                    w[2 * i + 1] = f.y;
                }
            }
#pragma unroll
            for (int o = 8; o; o >>= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
            const GroupParams p = group_params(mn, mx);
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = quantize_one(w[i], p);
            const uint32_t word = pack8(v);
            if (g < total_groups) {
                qw[g * 16 + sub] = word;
                if (sub == 0) {
                    scales[g] = __float2half_rn(p.s);
                    zeros[g] = static_cast<uint8_t>(p.zp);
                }
            }
        }
    }
}

}  // namespace w4
