// gemv.cuh -- W4A16 decode GEMV / skinny GEMM (M <= 8) on CUDA cores.
//
// Computes Y[m,n] = sum_k A[m,k] * (q[n,k] - zp[n,k/128]) * s16[n,k/128] with fp32
// accumulation ("Build a GPTQ INT4 Quantization Engine in Python/NumPy", Step 5, the
// fused dequantize-matmul; dequantization per "From Scratch: Building a GPTQ INT4
// Quantizer in Pure Python", Step 4).  Dequantization happens in registers; the
// fp16/bf16 weight matrix is never formed.
//
// Mapping: a warp owns R rows of W at a time and splits K across its lanes in
// 32-element chunks (16 packed bytes, always inside one 128-element group), so each
// lane reads one 16-byte word per row per step and the warp reads 512 contiguous
// bytes.  Per chunk the lane forms sum_k a_k * (q_k - zp) exactly-small-integer
// weighted in fp32, then scales by s once; partial sums meet in a xor-shuffle
// reduction at the end of the row (split-K inside the warp, no workspace).
#pragma once

#include "common.cuh"

namespace w4 {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&a)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[2 * i] = __uint_as_float(w[i] << 16);
        a[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <int MT, int R>
__global__ void __launch_bounds__(256) gemv_simple_kernel(
    const __nv_bfloat16 *__restrict__ A, const uint8_t *__restrict__ qweight,
    const __half *__restrict__ scales, const uint8_t *__restrict__ zeros,
    __nv_bfloat16 *__restrict__ Y, int64_t N, int64_t K) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t ng = K >> 7;
    const int64_t nchunk = K >> 5;
    const int64_t row_bytes = K >> 1;

    for (int64_t row0 = warp * R; row0 < N; row0 += nwarps * R) {
        float acc[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = 0.0f;

        for (int64_t c = lane; c < nchunk; c += 32) {
            const int64_t k0 = c << 5;
            const int64_t g = k0 >> 7;
            uint4 wq[R];
            float s[R], z[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r;
                if (row < N) {
                    wq[r] = ldg_stream_16(qweight + row * row_bytes + (c << 4));
                    s[r] = __half2float(scales[row * ng + g]);
                    z[r] = static_cast<float>(zeros[row * ng + g]);
                } else {
                    wq[r] = make_uint4(0, 0, 0, 0);
                    s[r] = 0.0f;
                    z[r] = 0.0f;
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 *ap = reinterpret_cast<const uint4 *>(A + m * K + k0);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float a[8];
                    bf16x8_to_f32(__ldg(ap + u), a);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t word = (u == 0) ? wq[r].x : (u == 1) ? wq[r].y
                                            : (u == 2) ? wq[r].z : wq[r].w;
                        float part = 0.0f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float qf = static_cast<float>((word >> (4 * i)) & 15u);
                            part = fmaf(a[i], qf - z[r], part);
                        }
                        acc[r][m] = fmaf(part, s[r], acc[r][m]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float v = acc[r][m];
#pragma unroll
                for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[r][m] = v;
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r;
                if (row < N) {
#pragma unroll
                    for (int m = 0; m < MT; ++m) Y[m * N + row] = __float2bfloat16_rn(acc[r][m]);
                }
            }
        }
    }
}

}  // namespace w4
