// gemv.cuh -- W4A16 decode GEMV / skinny GEMM (M <= 8) on CUDA cores.
//
// Computes Y[m,n] = sum_k A[m,k] * (q[n,k] - zp[n,k/128]) * s16[n,k/128] with fp32
// accumulation ("Build a GPTQ INT4 Quantization Engine in Python/NumPy", Step 5, the
// fused dequantize-matmul; dequantization per "From Scratch: Building a GPTQ INT4
// Quantizer in Pure Python", Step 4).  Dequantization happens in registers; the
// fp16/bf16 weight matrix is never formed.
//
// Streaming: each CTA owns a contiguous band of rows of W; a producer warp streams
// the band through a shared-memory ring of up to 8 stages (about 192 KB in flight per
// SM), one row per consumer warp per stage: the packed rows
// (contiguous in memory) with one 1-D bulk copy (cp.async.bulk) and their scales and
// zero points with two 2-D tensor copies, all completing on the stage's mbarrier.
// Consumer warps take one row each per stage; the lanes of a warp split K
// (split-K inside the warp; partial sums meet in a xor-shuffle reduction, no
// workspace).  With M * (K / 4096) <= 2 the activations live in registers (lane =
// 128-group); otherwise in shared memory (lane = 32-element chunk).
//
// Arithmetic per chunk, for each activation row m:
//   v_k   = bf16(128 + q_k): the nibble ORed into the bf16 pattern of 128 (ulp 1),
//           two levels per lop3 (pairs (k, k+4) of each 8-level word)
//   acc   = sum_k a_k * v_k, fp32, with fma.rn.f32.bf16 (exact products, one
//           rounding per term; activations are read from shared memory already
//           permuted into the same (k, k+4) pairs)
//   part += s * (acc - (128 + zp) * SA)
// where SA = (sum_k a_k) is precomputed per chunk with the very same fma chain run
// on v_k = 128 and scaled by 1/128 (exact).  Hence a chunk whose levels all equal
// zp = 0 (the only way a group reconstructs to all zeros) contributes exactly 0, and
// otherwise the correction's rounding stays near 2^-24 relative to the terms.
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

// Fallback for shapes whose activations do not fit in shared memory: a warp owns R
// rows, lanes split K in 32-element chunks, activations are read from global memory.
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

namespace gemv {

constexpr int MAX_STAGES = 8;
constexpr int RING_BYTES = 192 * 1024;                     // target bytes in flight per SM
constexpr uint32_t kMagic128x2 = 0x43004300u;              // bf16 pair (128, 128)
// Consumer warps (= rows per stage, one row per warp) of each kernel; plus one
// producer warp.
constexpr int CW_REGA = 16;   // activations in registers, 64 per lane
constexpr int CW_SMEMA = 8;   // activations in shared memory, or 128 registers per lane
__host__ __device__ constexpr int num_threads(int cw) { return (cw + 1) * 32; }

struct Params {
    const __nv_bfloat16 *A;
    const uint8_t *qweight;
    __nv_bfloat16 *Y;
    int N, K;
    int rows_per_cta;     // band size (the last CTA may get fewer)
    int stages;           // ring depth (<= MAX_STAGES)
    WaitParams wait;
};

// acc + a.lo * b.lo + a.hi * b.hi: two chained mixed-precision fp32 FMAs on bf16
// halves (exact products, each addition rounded once).
__device__ __forceinline__ float fma_bf16x2(uint32_t a2, uint32_t b2, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 t;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 t, al, bl, %3;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, t;\n\t}"
        : "=f"(d)
        : "r"(a2), "r"(b2), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;  // (a & b) | c
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Packed word (8 levels, element i in bits [4i, 4i+4)) -> bf16 pairs (128 + q_j,
// 128 + q_{j+4}) for j = 0..3.
__device__ __forceinline__ void levels_to_bf16(uint32_t x, uint32_t *v) {
    const uint32_t mask = 0x000F000Fu;
    v[0] = lop3_and_or(x, mask, kMagic128x2);
    v[1] = lop3_and_or(x >> 4, mask, kMagic128x2);
    v[2] = lop3_and_or(x >> 8, mask, kMagic128x2);
    v[3] = lop3_and_or(x >> 12, mask, kMagic128x2);
}

// The fp32 chain over one 32-element chunk: v[16] level pairs (4 per packed word),
// a[4] activation pieces (4 pair-words each).  Two interleaved accumulators.
__device__ __forceinline__ float chunk_dot(const uint32_t (&v)[16], const uint4 (&a)[4]) {
    float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc0 = fma_bf16x2(a[i].x, v[4 * i + 0], acc0);
        acc1 = fma_bf16x2(a[i].y, v[4 * i + 1], acc1);
        acc0 = fma_bf16x2(a[i].z, v[4 * i + 2], acc0);
        acc1 = fma_bf16x2(a[i].w, v[4 * i + 3], acc1);
    }
    return __fadd_rn(acc0, acc1);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// 8 consecutive bf16 (natural order, one 16-byte piece) -> (k, k+4) pairs.
__device__ __forceinline__ uint4 pair_permute(uint4 nat) {
    uint4 pr;
    pr.x = prmt(nat.x, nat.z, 0x5410u);
    pr.y = prmt(nat.x, nat.z, 0x7632u);
    pr.z = prmt(nat.y, nat.w, 0x5410u);
    pr.w = prmt(nat.y, nat.w, 0x7632u);
    return pr;
}

// Stage layout in shared memory (all pieces 128-byte aligned), R rows per stage:
//   W rows  R x K/2 bytes     (1-D bulk copy; row-contiguous)
//   scales  R x ng fp16       (2-D tensor copy, box {ng, R})
//   zeros   R x ng uint8      (2-D tensor copy, box {ng, R})
__host__ __device__ inline int up128(int x) { return (x + 127) / 128 * 128; }
__host__ __device__ inline int stage_off_s(int K, int R) { return up128(R * (K / 2)); }
__host__ __device__ inline int stage_off_z(int K, int R) { return stage_off_s(K, R) + up128(R * (K / 128) * 2); }
__host__ __device__ inline int stage_bytes(int K, int R) { return stage_off_z(K, R) + up128(R * (K / 128)); }

// ---- producer warp: W rows + scales + zeros of each stage ---------------------------
template <int R>
__device__ __forceinline__ void produce(const Params &p, const CUtensorMap *tmS, const CUtensorMap *tmZ,
                                        uint8_t *ring, uint64_t *full, uint64_t *empty,
                                        volatile int *abort_flag, int n_begin, int n_end,
                                        int num_stages) {
    const int lane = lane_id();
    if (lane != 0) return;
    const int K = p.K, ng = K / 128, row_bytes = K / 2;
    const int sb = stage_bytes(K, R);
    const int off_s = stage_off_s(K, R);
    const int off_z = stage_off_z(K, R);
    const int S = p.stages;
    const uint64_t pol_w = policy_evict_first(), pol_sz = policy_evict_first();
    const unsigned long long tmo = p.wait.timeout_ns;
    int issued_parity[MAX_STAGES];
#pragma unroll
    for (int s = 0; s < MAX_STAGES; ++s) issued_parity[s] = -1;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int i = 0; i < num_stages; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, tmo)) {
            ok = false;
            break;
        }
        const int r0 = n_begin + i * R;
        const int rows = min(R, n_end - r0);
        const uint32_t wbytes = static_cast<uint32_t>(rows) * row_bytes;
        uint8_t *st = ring + static_cast<size_t>(stage) * sb;
        mbar_arrive_expect_tx(&full[stage], wbytes + R * ng * 3);
        bulk_copy_g2s(st, p.qweight + static_cast<int64_t>(r0) * row_bytes, wbytes, &full[stage], pol_w);
        tma_load_2d(st + off_s, tmS, &full[stage], 0, r0, pol_sz);
        tma_load_2d(st + off_z, tmZ, &full[stage], 0, r0, pol_sz);
#pragma unroll
        for (int s = 0; s < MAX_STAGES; ++s)
            if (s == static_cast<int>(stage)) issued_parity[s] = static_cast<int>(phase);
        if (++stage == static_cast<uint32_t>(S)) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (!ok) {
        // Every copy this thread issued must land before the CTA exits.
        const unsigned long long t0 = globaltimer_ns();
#pragma unroll
        for (int s = 0; s < MAX_STAGES; ++s) {
            if (issued_parity[s] < 0) continue;
            while (!mbar_try_wait(smem_addr(&full[s]), static_cast<uint32_t>(issued_parity[s])))
                if (globaltimer_ns() - t0 > tmo) break;
        }
    }
}

// Converts a stored fp16 scale / uint8 zero point to (scale, 128 + zp) in fp32.
__device__ __forceinline__ float scale_f32(unsigned short s16) {
    float r;
    asm("{\n\t.reg .b16 h;\n\tmov.b16 h, %1;\n\tadd.rn.f32.f16 %0, h, 0f80000000;\n\t}" : "=f"(r) : "h"(s16));
    return r;
}
__device__ __forceinline__ float zero_plus_128(uint32_t z) {
    return __fsub_rn(__uint_as_float(0x4B000000u + 128u + z), 8388608.0f);
}

__device__ __forceinline__ bool warp_wait_full(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                               unsigned long long tmo) {
    int got = 1;
    if (lane_id() == 0) got = mbar_wait(bar, parity, abort_flag, tmo) ? 1 : 0;
    got = __shfl_sync(0xffffffffu, got, 0);
    __syncwarp();
    return got != 0;
}

__device__ __forceinline__ void stall_hook(const Params &p, uint64_t *never, volatile int *abort_flag, bool &ok) {
    if (ok && p.wait.stall) {  // test hook: wait on a barrier that nothing signals
        ok = warp_wait_full(never, 0, abort_flag, p.wait.timeout_ns);
    }
}

// ======================================================================================
// Activations in registers (MT * GPL <= 2): lane l owns groups l + 32 i (i < GPL) of
// every row and keeps those groups' activations, pair-permuted, in registers.  Per row
// it reads its 64 packed bytes per group as four 16-byte pieces in a lane-rotated order
// (piece (j + l/2) & 3 at step j), which keeps the quarter-warp reads conflict-free;
// the registers were loaded in the same rotation.
// ======================================================================================
template <int MT, int GPL, int CW>
__global__ void __launch_bounds__(num_threads(CW), 1)
    gemv_rega_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                     const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int R = CW;  // rows per stage
    const int K = p.K, ng = K >> 7, row_bytes = K >> 1;
    const int S = p.stages;
    const int sb = stage_bytes(K, R);
    const int off_s = stage_off_s(K, R);
    const int off_z = stage_off_z(K, R);
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + static_cast<size_t>(S) * sb);
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *never = empty + MAX_STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(never + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long tmo = p.wait.timeout_ns;
    const int n_begin = blockIdx.x * p.rows_per_cta;
    const int n_end = min(p.N, n_begin + p.rows_per_cta);
    const int band = max(0, n_end - n_begin);
    const int num_stages = (band + R - 1) / R;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmS);
        prefetch_tensormap(&tmZ);
    }
    __syncthreads();

    if (warp == CW) {
        produce<R>(p, &tmS, &tmZ, ring, full, empty, abort_flag, n_begin, n_end, num_stages);
        __syncwarp();
    } else {
        const int rot = lane >> 1;
        // Activations of my groups, pair-permuted, in rotated piece order, and their
        // chain sums SA = chain(a, 128) / 128 (bit-identical to the per-row chain).
        uint4 a[MT][GPL][4][4];
        float sa[MT][GPL];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int i = 0; i < GPL; ++i) {
                const int g = lane + 32 * i;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int piece = (j + rot) & 3;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint4 nat = make_uint4(0, 0, 0, 0);
                        if (g < ng)
                            nat = __ldg(reinterpret_cast<const uint4 *>(
                                p.A + static_cast<int64_t>(m) * K + g * 128 + piece * 32 + u * 8));
                        a[m][i][j][u] = pair_permute(nat);
                    }
                }
            }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int i = 0; i < GPL; ++i) {
                uint32_t v[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = kMagic128x2;
                float tot = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) tot = __fadd_rn(tot, chunk_dot(v, a[m][i][j]));
                sa[m][i] = tot * 0.0078125f;
            }

        bool ok = true;
        stall_hook(p, never, abort_flag, ok);
        uint32_t stage = 0, phase = 0;
        for (int it = 0; ok && it < num_stages; ++it) {
            if (!warp_wait_full(&full[stage], phase, abort_flag, tmo)) break;
            const int r0 = n_begin + it * R;
            const int rows = min(R, n_end - r0);
            const uint8_t *st = smem + static_cast<size_t>(stage) * sb;
            const int rl = warp;  // one row per warp per stage
            if (rl < rows) {
                const unsigned short *srow = reinterpret_cast<const unsigned short *>(st + off_s) + rl * ng;
                const uint8_t *zrow = st + off_z + rl * ng;
                float y[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) y[m] = 0.0f;
#pragma unroll
                for (int i = 0; i < GPL; ++i) {
                    const int g = lane + 32 * i;
                    if (g < ng) {
                        const float sf = scale_f32(srow[g]);
                        const float zf = zero_plus_128(zrow[g]);
                        const uint4 *wrow = reinterpret_cast<const uint4 *>(st + rl * row_bytes + g * 64);
                        const uint4 w0 = wrow[rot & 3], w1 = wrow[(1 + rot) & 3];
                        const uint4 w2 = wrow[(2 + rot) & 3], w3 = wrow[(3 + rot) & 3];
                        float part[MT];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {   // half a group at a time
                            uint32_t v[2][16];
                            const uint4 wa = h ? w2 : w0, wb = h ? w3 : w1;
                            levels_to_bf16(wa.x, v[0]);
                            levels_to_bf16(wa.y, v[0] + 4);
                            levels_to_bf16(wa.z, v[0] + 8);
                            levels_to_bf16(wa.w, v[0] + 12);
                            levels_to_bf16(wb.x, v[1]);
                            levels_to_bf16(wb.y, v[1] + 4);
                            levels_to_bf16(wb.z, v[1] + 8);
                            levels_to_bf16(wb.w, v[1] + 12);
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                const float c0 = chunk_dot(v[0], a[m][i][2 * h]);
                                const float c1 = chunk_dot(v[1], a[m][i][2 * h + 1]);
                                part[m] = h ? __fadd_rn(__fadd_rn(part[m], c0), c1)
                                            : __fadd_rn(__fadd_rn(0.0f, c0), c1);
                            }
                        }
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const float t = __fsub_rn(part[m], __fmul_rn(zf, sa[m][i]));
                            y[m] = __fmaf_rn(sf, t, y[m]);
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
#pragma unroll
                    for (int o = 16; o; o >>= 1) y[m] += __shfl_xor_sync(0xffffffffu, y[m], o);
                }
                if (lane < MT) {
                    float out = y[0];
#pragma unroll
                    for (int m = 1; m < MT; ++m)
                        if (lane == m) out = y[m];
                    p.Y[static_cast<int64_t>(lane) * p.N + r0 + rl] = __float2bfloat16_rn(out);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == static_cast<uint32_t>(S)) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    __syncthreads();
}

// ======================================================================================
// Activations in shared memory (any MT <= 8): lane l owns the 16-byte chunks
// c = l + 32 j of each row (32 levels, inside one group).  The activations arrive by
// one bulk copy and are rearranged in place: piece i (elements 8i..8i+7) of chunk c
// holds (k, k+4) pairs and sits at slot i ^ ((c >> 1) & 3), so the lanes' reads of
// consecutive chunks are conflict-free.
// ======================================================================================
__host__ __device__ inline size_t smem_bytes_smema(int MT, int K, int stages) {
    const size_t nchunk = static_cast<size_t>(K) / 32;
    return static_cast<size_t>(stages) * stage_bytes(K, CW_SMEMA) + static_cast<size_t>(MT) * K * 2 +
           MT * nchunk * 4 + (2 * MAX_STAGES + 2) * 8 + 16;
}
__host__ __device__ inline size_t smem_bytes_rega(int K, int stages, int cw) {
    return static_cast<size_t>(stages) * stage_bytes(K, cw) + (2 * MAX_STAGES + 1) * 8 + 16;
}

__device__ __forceinline__ uint32_t a_slot(int c, int i) { return static_cast<uint32_t>(i ^ ((c >> 1) & 3)); }

template <int MT, int CW>
__global__ void __launch_bounds__(num_threads(CW), 1)
    gemv_smema_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                      const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int R = CW;
    const int K = p.K, ng = K >> 7, row_bytes = K >> 1, nchunk = K >> 5;
    const int S = p.stages;
    const int sb = stage_bytes(K, R);
    const int off_s = stage_off_s(K, R);
    const int off_z = stage_off_z(K, R);
    uint8_t *ring = smem;
    uint4 *a_sm = reinterpret_cast<uint4 *>(smem + static_cast<size_t>(S) * sb);
    float *sa = reinterpret_cast<float *>(a_sm + static_cast<size_t>(MT) * 4 * nchunk);
    uint64_t *full = reinterpret_cast<uint64_t *>(sa + static_cast<size_t>(MT) * nchunk);
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *a_bar = empty + MAX_STAGES;
    uint64_t *never = a_bar + 1;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(never + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long tmo = p.wait.timeout_ns;
    const int n_begin = blockIdx.x * p.rows_per_cta;
    const int n_end = min(p.N, n_begin + p.rows_per_cta);
    const int band = max(0, n_end - n_begin);
    const int num_stages = (band + R - 1) / R;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        mbar_init(a_bar, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmS);
        prefetch_tensormap(&tmZ);
    }
    __syncthreads();

    if (warp == CW) {
        if (lane == 0) {
            const uint32_t abytes = static_cast<uint32_t>(MT) * row_bytes * 4;  // MT * K * 2
            mbar_arrive_expect_tx(a_bar, abytes);
            bulk_copy_g2s(a_sm, p.A, abytes, a_bar, policy_evict_last());
        }
        produce<R>(p, &tmS, &tmZ, ring, full, empty, abort_flag, n_begin, n_end, num_stages);
        if (lane == 0) {  // the activation copy must land before the CTA exits
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_addr(a_bar), 0))
                if (globaltimer_ns() - t0 > tmo) break;
        }
        __syncwarp();
    } else {
        bool ok = warp_wait_full(a_bar, 0, abort_flag, tmo);
        for (int t = threadIdx.x; ok && t < MT * nchunk; t += CW * 32) {
            const int c = t % nchunk;
            uint4 *chunk = a_sm + static_cast<size_t>(t) * 4;
            uint4 nat[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) nat[i] = chunk[i];
#pragma unroll
            for (int i = 0; i < 4; ++i) chunk[a_slot(c, i)] = pair_permute(nat[i]);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory");
        for (int t = threadIdx.x; ok && t < MT * nchunk; t += CW * 32) {
            const int c = t % nchunk;
            const uint4 *chunk = a_sm + static_cast<size_t>(t) * 4;
            uint4 a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = chunk[a_slot(c, i)];
            uint32_t v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = kMagic128x2;
            sa[t] = chunk_dot(v, a) * 0.0078125f;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory");

        stall_hook(p, never, abort_flag, ok);
        uint32_t stage = 0, phase = 0;
        for (int it = 0; ok && it < num_stages; ++it) {
            if (!warp_wait_full(&full[stage], phase, abort_flag, tmo)) break;
            const int r0 = n_begin + it * R;
            const int rows = min(R, n_end - r0);
            const uint8_t *st = smem + static_cast<size_t>(stage) * sb;
            const int rl = warp;
            if (rl < rows) {
                const unsigned short *srow = reinterpret_cast<const unsigned short *>(st + off_s) + rl * ng;
                const uint8_t *zrow = st + off_z + rl * ng;
                float y[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) y[m] = 0.0f;
#pragma unroll 2
                for (int c = lane; c < nchunk; c += 32) {
                    const float sf = scale_f32(srow[c >> 2]);
                    const float zf = zero_plus_128(zrow[c >> 2]);
                    const uint4 w = *reinterpret_cast<const uint4 *>(st + rl * row_bytes + c * 16);
                    uint32_t v[16];
                    levels_to_bf16(w.x, v);
                    levels_to_bf16(w.y, v + 4);
                    levels_to_bf16(w.z, v + 8);
                    levels_to_bf16(w.w, v + 12);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint4 *chunk = a_sm + (static_cast<size_t>(m) * nchunk + c) * 4;
                        uint4 a[4];
#pragma unroll
                        for (int i2 = 0; i2 < 4; ++i2) a[i2] = chunk[a_slot(c, i2)];
                        const float acc = chunk_dot(v, a);
                        const float t = __fsub_rn(acc, __fmul_rn(zf, sa[m * nchunk + c]));
                        y[m] = __fmaf_rn(sf, t, y[m]);
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
#pragma unroll
                    for (int o = 16; o; o >>= 1) y[m] += __shfl_xor_sync(0xffffffffu, y[m], o);
                }
                if (lane < MT) {
                    float out = y[0];
#pragma unroll
                    for (int m = 1; m < MT; ++m)
                        if (lane == m) out = y[m];
                    p.Y[static_cast<int64_t>(lane) * p.N + r0 + rl] = __float2bfloat16_rn(out);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == static_cast<uint32_t>(S)) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    __syncthreads();
}

}  // namespace gemv
}  // namespace w4
