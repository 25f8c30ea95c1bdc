// dequantize.cuh -- materialize W_hat[N,K] = (q - zp) * s16 as a bf16 or fp16 tensor.
//
// Method ("From Scratch: Building a GPTQ INT4 Quantizer in Pure Python", Step 4:
// dequantize = (q - zero_point) * scale): per level, with q the 4-bit level, zp the
// group's zero point and s16 its fp16 scale, the product (q - zp) * s16 is exact in
// fp32 (a 5-bit integer times an 11-bit significand), so it is formed exactly and
// rounded once to the output type (round to nearest even; fp16 overflows to +-inf).
//
// HBM-bound: 0.5 byte read and 2 bytes written per level (plus 3 bytes per group of
// scales and zero points).  The tensor is walked as one flat array of levels (groups
// never straddle rows because K is a multiple of 128): a thread takes 8 consecutive
// levels (4 packed bytes -> 16 output bytes), so a warp reads 128 contiguous bytes and
// writes 512 contiguous bytes per step, and 16 consecutive threads share a group's
// scale and zero point (broadcast loads).  Grid-stride over the chunks, eight chunks in
// flight per thread; outputs are written with streaming stores (they are not re-read).
// Exact level arithmetic: the even and odd levels of a word are split with two masks,
// one prmt per level places a level under the exponent byte of 2^23 (giving the float
// 2^23 + q), minus (2^23 + zp) gives q - zp exactly and times s16 is exact; both are
// done two levels at a time in f32x2.
#pragma once

#include "common.cuh"

namespace w4 {
namespace deq {

constexpr int NUM_THREADS = 256;
constexpr int UNROLL = 8;                     // chunks in flight per thread
constexpr int BLOCKS_PER_SM = 8;

__device__ __forceinline__ uint32_t ldg_nc_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
    uint32_t r;
    if (bf16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// 8 levels of one packed word (level i in bits [4i, 4i+4)) -> 8 outputs, element i in
// the low half of word i/2 when i is even.
template <bool kBF16>
__device__ __forceinline__ uint4 dequant_chunk(uint32_t x, float s, float m) {
    const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;   // levels 2b / 2b+1 in byte b
    const uint32_t M = 0x4B000000u;                                     // 2^23
    uint64_t m2, s2;
    asm("mov.b64 %0, {%1, %1};" : "=l"(m2) : "f"(m));
    asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(s));
    uint32_t w[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        // byte b of lo / hi as the low byte, bytes 0, 0, 0x4B above it: 2^23 + q
        const uint32_t t0 = prmt(lo, M, 0x7540u + b), t1 = prmt(hi, M, 0x7540u + b);
        uint64_t v;
        asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(t0), "r"(t1));
        asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(v) : "l"(v), "l"(m2));   // q - zp, exact
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(v) : "l"(v), "l"(s2));   // (q - zp) * s16, exact
        float v0, v1;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(v0), "=f"(v1) : "l"(v));
        w[b] = pack2(v0, v1, kBF16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void st_stream_16(uint4 *p, uint4 v) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

template <bool kBF16>
__global__ void __launch_bounds__(NUM_THREADS)
    dequantize_kernel(const uint32_t *__restrict__ qw, const __half *__restrict__ scales,
                      const uint8_t *__restrict__ zeros, uint4 *__restrict__ out, int64_t chunks) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * NUM_THREADS;
    for (int64_t c0 = static_cast<int64_t>(blockIdx.x) * NUM_THREADS + threadIdx.x; c0 < chunks;
         c0 += stride * UNROLL) {
        uint32_t x[UNROLL];
        float s[UNROLL], m[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t c = c0 + u * stride;
            x[u] = 0u;
            s[u] = 0.0f;
            m[u] = 8388608.0f;
            if (c < chunks) {
                const int64_t g = c >> 4;                                   // 16 chunks per group
                x[u] = ldg_nc_u32(qw + c);
                s[u] = __half2float(scales[g]);
                m[u] = __uint_as_float(0x4B000000u | zeros[g]);             // 2^23 + zp, exact
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t c = c0 + u * stride;
            if (c < chunks) st_stream_16(out + c, dequant_chunk<kBF16>(x[u], s[u], m[u]));
        }
    }
}

}  // namespace deq
}  // namespace w4
