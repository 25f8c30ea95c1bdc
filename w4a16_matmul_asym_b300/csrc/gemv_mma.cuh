// gemv_mma.cuh -- W4A16 decode GEMV / skinny GEMM (1 <= M <= 16) on warp-level
// tensor-core MMAs, with the weights dequantized in registers.
//
// Computes Y[m,n] = sum_g s16[n,g] * sum_{k in g} A[m,k] * (q[n,k] - zp[n,g]) with fp32
// accumulation: "Build a GPTQ INT4 Quantization Engine in Python/NumPy", Step 5 (the
// fused dequantize-matmul over packed weights), dequantization as in "From Scratch:
// Building a GPTQ INT4 Quantizer in Pure Python", Step 4 ((q - zero_point) * scale).
// Neither the fp16/bf16 weight matrix nor a dequantized tile ever reaches memory.
//
// Why warp MMAs here.  A decode step reads 0.52 bytes per weight and must consume
// ~44 weights per clock per SM to keep up with HBM.  On the CUDA cores every weight
// costs M multiply-adds (8 at M = 8), which caps the M = 8 case far below bandwidth.
// tcgen05 MMAs read their weight operand from shared or tensor memory, so the
// dequantized bf16 tile would have to be written there and read back (4 bytes of
// shared-memory traffic per weight, above the 128 B/clk an SM has at that rate).
// mma.sync takes its A fragment straight from registers: each thread turns its
// packed levels into bf16 pairs and hands them to the tensor core, and one MMA
// (16 weight rows x 16 k) serves up to 8 activation rows (16 with two MMAs).
//
// Data movement.  A tile is 16 rows of W; CTA c owns a contiguous range of tiles (one
// CTA per SM).  A stage is one tile's 2048-wide k-slice (16 groups), brought in by three
// tensor copies that complete on the stage's mbarrier: the packed levels through a 3-D
// tensor map that views qweight as (64 bytes of a group, row, group), so the 16 KB land
// group-major ([group][row][64 B]: each consumer warp's group is one contiguous 1 KB
// block, and the 8 lanes of a quarter warp read 128 contiguous bytes); the 16 x 16
// scales and zero points through 2-D maps.  Rows past N are zero-filled by the copy.
// Up to MAX_STAGES stages are in flight.  The activations are copied once per CTA into
// shared memory, permuted so that every B fragment is one conflict-free 16-byte load.
//
// Work split.  Consumer warp w takes quantization group w of every stage (the 16
// groups of a 2048-wide slice), i.e. split-K across the 16 warps; its partial sums of
// a tile stay in registers across the tile's stages and go to a double-buffered
// reduction area at the tile's end; an epilogue warp adds the 16 partials in a fixed
// order (deterministic), rounds to bf16 and stores Y.
//
// Fragment mapping (m16n8k16, A row-major = W rows, B column-major = activation rows):
// lane (g, t) = (lane / 4, lane % 4) holds W rows g and g + 8 and, of each group, the
// 32 levels k = 32 t .. 32 t + 31 (one 16-byte load per row).  Packed word v (levels
// 8v .. 8v+7 of that range) becomes four bf16 pairs (k, k+4) for k = 0..3 of the word;
// MMA (v, 0) takes the pairs (0,4), (1,5) as logical columns (2t, 2t+1), (2t+8, 2t+9)
// and MMA (v, 1) the pairs (2,6), (3,7).  Over the 8 MMAs of a group every k is used
// once; the activations are stored in the same pairing, so B fragments match.
//
// Dequantization, exact: lop3 puts a level into the low mantissa bits of bf16(128),
// giving bf16(128 + q) (ulp 1 there), two levels per instruction; sub.bf16x2 of
// bf16(128 + zp) gives q - zp exactly (an integer in [-15, 15]).  The MMA sums exact
// products in fp32; the group's sum is scaled by the fp32 value of s16 and added to
// the running fp32 sum: all-zero groups contribute exactly 0.
#pragma once

#include "common.cuh"
#include "gemm_tcgen05.cuh"   // tensor-map encoding (driver entry point)

namespace w4 {
namespace gmma {

constexpr int CW = 16;                        // consumer warps = groups per stage
constexpr int PRODUCER = CW;                  // warp index of the producer
constexpr int EPILOGUE = CW + 1;              // warp index of the epilogue
constexpr int NUM_THREADS = (CW + 2) * 32;
constexpr int ROWS = 16;                      // W rows per tile (the MMA's M)
constexpr int KC = CW * 128;                  // k per stage
constexpr int GROUP_BYTES = 64;               // packed bytes of one group of one row
constexpr int SLOT_W = CW * ROWS * GROUP_BYTES;  // [group][row][64 B]
constexpr int SLOT_S = ROWS * CW * 2;         // fp16 scales [row][group]
constexpr int SLOT_Z = ROWS * CW;             // uint8 zero points [row][group]
constexpr int SLOT_BYTES = SLOT_W + SLOT_S + SLOT_Z;
constexpr int MAX_STAGES = 12;
constexpr int RED_STRIDE = 20;                // floats per (warp, column): conflict-free writes
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr uint32_t kBf16x2_128 = 0x43004300u;  // bf16 pair (128, 128)

__host__ __device__ constexpr int red_bytes(int nb) { return 2 * CW * 8 * nb * RED_STRIDE * 4; }
__host__ __device__ constexpr int a_bytes(int M, int K) { return (M * K * 2 + 127) / 128 * 128; }
__host__ __device__ constexpr int bar_bytes() { return (2 * MAX_STAGES + 5) * 8 + 16; }
__host__ __device__ constexpr int smem_bytes(int M, int K, int nb, int stages) {
    return a_bytes(M, K) + stages * SLOT_BYTES + red_bytes(nb) + bar_bytes();
}

struct Params {
    const __nv_bfloat16 *A;   // [M, K]
    const uint8_t *qweight;   // [N, K/2]
    const __half *scales;     // [N, K/128]
    const uint8_t *zeros;     // [N, K/128]
    __nv_bfloat16 *Y;         // [M, N]
    int M, N, K;
    int tiles;                // ceil(N / 16)
    int stages;               // ring depth (<= MAX_STAGES)
    WaitParams wait;
};

// ---- small device helpers -------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// 8 consecutive bf16 (one 16-byte piece, natural order) -> (k, k+4) pairs:
// [a0 a4 a1 a5 a2 a6 a3 a7].
__device__ __forceinline__ uint4 pair_permute(const uint4 &nat) {
    uint4 r;
    r.x = prmt(nat.x, nat.z, 0x5410u);
    r.y = prmt(nat.x, nat.z, 0x7632u);
    r.z = prmt(nat.y, nat.w, 0x5410u);
    r.w = prmt(nat.y, nat.w, 0x7632u);
    return r;
}
// (x & 0x000F000F) | bf16x2(128, 128): levels at bits [0,4) and [16,20) -> bf16(128 + q).
__device__ __forceinline__ uint32_t level_pair(uint32_t x) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(0x000F000Fu), "r"(kBf16x2_128));
    return d;
}
__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// d += A(16x16, bf16) * B(16x8, bf16), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
    float r;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.f32.f16 %0, t;\n\t}" : "=f"(r) : "r"(h));
    return r;
}
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// One lane waits (bounded), the warp follows its verdict.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned long long tmo, bool polite) {
    int got = 1;
    if (lane_id() == 0)
        got = (polite ? mbar_wait_polite(bar, parity, abort_flag, tmo) : mbar_wait(bar, parity, abort_flag, tmo))
                  ? 1 : 0;
    got = __shfl_sync(0xffffffffu, got, 0);
    __syncwarp();
    return got != 0;
}

// ---- producer warp ----------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t x,
                                            int32_t y, int32_t z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// One thread issues every stage: three tensor copies (x coordinates 0 and 16 ks, both
// multiples of 16 bytes).
__device__ __forceinline__ void produce(const Params &p, const CUtensorMap *tmW, const CUtensorMap *tmS,
                                        const CUtensorMap *tmZ, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                        volatile int *abort_flag, int t_begin, int nstages) {
    if (lane_id() != 0) return;
    const int KS = p.K / KC, S = p.stages;
    const unsigned long long tmo = p.wait.timeout_ns;
    const uint64_t pol = policy_evict_first();
    uint32_t slot = 0, phase = 0;
    int issued = 0;
    bool ok = true;
    for (int i = 0; i < nstages; ++i) {
        if (!mbar_wait_polite(&empty[slot], phase ^ 1u, abort_flag, tmo)) {
            ok = false;
            break;
        }
        const int tile = t_begin + i / KS, ks = i % KS;
        const int n0 = tile * ROWS;
        uint8_t *st = ring + static_cast<size_t>(slot) * SLOT_BYTES;
        mbar_arrive_expect_tx(&full[slot], SLOT_BYTES);
        tma_load_3d(st, tmW, &full[slot], 0, n0, ks * CW, pol);
        tma_load_2d(st + SLOT_W, tmS, &full[slot], ks * CW, n0, pol);
        tma_load_2d(st + SLOT_W + SLOT_S, tmZ, &full[slot], ks * CW, n0, pol);
        ++issued;
        if (++slot == static_cast<uint32_t>(S)) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (!ok) {
        // Every copy issued must land before the CTA exits: wait (bounded) for the
        // last min(issued, S) stages' barriers.
        const unsigned long long t0 = globaltimer_ns();
        const int first = issued > S ? issued - S : 0;
        for (int i = first; i < issued; ++i) {
            const uint32_t par = static_cast<uint32_t>((i / S) & 1);
            while (!mbar_try_wait(smem_addr(&full[i % S]), par))
                if (globaltimer_ns() - t0 > tmo) break;
        }
    }
}

// ---- epilogue warp -------------------------------------------------------------------------
template <int NB>
__device__ __forceinline__ void epilogue(const Params &p, const float *red, uint64_t *red_full, uint64_t *red_empty,
                                         volatile int *abort_flag, int t_begin, int ntiles) {
    constexpr int COLS = 8 * NB;
    const int lane = lane_id();
    const int r = lane & 15;
    const unsigned long long tmo = p.wait.timeout_ns;
    for (int j = 0; j < ntiles; ++j) {
        const int b = j & 1;
        if (!warp_wait(&red_full[b], static_cast<uint32_t>((j >> 1) & 1), abort_flag, tmo, true)) return;
        const float *rb = red + b * CW * COLS * RED_STRIDE;
        float acc[COLS / 2];
#pragma unroll
        for (int i = 0; i < COLS / 2; ++i) {
            const int m = (lane >> 4) + 2 * i;
            float a = 0.0f;
#pragma unroll
            for (int w = 0; w < CW; ++w) a = __fadd_rn(a, rb[(w * COLS + m) * RED_STRIDE + r]);
            acc[i] = a;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[b]);
        const int n = (t_begin + j) * ROWS + r;
        if (n < p.N) {
#pragma unroll
            for (int i = 0; i < COLS / 2; ++i) {
                const int m = (lane >> 4) + 2 * i;
                if (m < p.M) p.Y[static_cast<int64_t>(m) * p.N + n] = __float2bfloat16_rn(acc[i]);
            }
        }
    }
}

// ---- the kernel ----------------------------------------------------------------------------
// NB = number of 8-column activation blocks (1: M <= 8, 2: M <= 16).
template <int NB>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmZ, const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int COLS = 8 * NB;
    const int M = p.M, K = p.K;
    const int KS = K / KC;
    const int S = p.stages;
    uint8_t *ring = smem + a_bytes(M, K);
    float *red = reinterpret_cast<float *>(ring + static_cast<size_t>(S) * SLOT_BYTES);
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(red) + red_bytes(NB));
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *red_full = empty + MAX_STAGES;
    uint64_t *red_empty = red_full + 2;
    uint64_t *never = red_empty + 2;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(never + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned long long tmo = p.wait.timeout_ns;
    const int t_begin = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.tiles / gridDim.x);
    const int t_end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.tiles / gridDim.x);
    const int ntiles = t_end - t_begin;
    const int nstages = ntiles * KS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&red_full[b], CW);
            mbar_init(&red_empty[b], 1);
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmS);
        prefetch_tensormap(&tmZ);
    }
    __syncthreads();

    if (warp == PRODUCER) {
        produce(p, &tmW, &tmS, &tmZ, ring, full, empty, abort_flag, t_begin, nstages);
        return;
    }
    if (warp == EPILOGUE) {
        epilogue<NB>(p, red, red_full, red_empty, abort_flag, t_begin, ntiles);
        return;
    }

    // ---- consumers: stage the activations, permuted: the 16-byte chunk (g, v, m, t)
    // (index ((4 g + v) M + m) 4 + t) holds A[m, 128 g + 32 t + 8 v + (0 4 1 5 2 6 3 7)].
    // Threads walk the chunks in shared-memory order, so the stores are conflict-free.
    const uint32_t a_base = smem_addr(smem);
    {
        const int total = M * (K >> 3);
        constexpr int BATCH = 8;
        for (int c0 = threadIdx.x; c0 < total; c0 += BATCH * CW * 32) {
            uint4 nat[BATCH];
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int c = c0 + u * CW * 32;
                nat[u] = make_uint4(0, 0, 0, 0);
                if (c < total) {
                    const int t = c & 3, rest = c >> 2;
                    const int m = rest % M, gv = rest / M;
                    const int g = gv >> 2, v = gv & 3;
                    nat[u] = __ldg(reinterpret_cast<const uint4 *>(p.A + static_cast<int64_t>(m) * K + g * 128 +
                                                                   t * 32 + v * 8));
                }
            }
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int c = c0 + u * CW * 32;
                if (c < total) sts128(a_base + (static_cast<uint32_t>(c) << 4), pair_permute(nat[u]));
            }
        }
    }
    named_barrier_sync(1, CW * 32);

    bool ok = true;
    if (p.wait.stall) ok = warp_wait(never, 0, abort_flag, tmo, false);  // test hook

    const int g8 = lane >> 2, t4 = lane & 3;
    const uint32_t ring_base = smem_addr(ring);
    const uint32_t w_off0 = warp * (ROWS * GROUP_BYTES) + g8 * GROUP_BYTES + t4 * 16;
    const uint32_t w_off1 = w_off0 + 8 * GROUP_BYTES;
    const uint32_t s_off0 = SLOT_W + g8 * (CW * 2) + warp * 2;
    const uint32_t s_off1 = s_off0 + 8 * (CW * 2);
    const uint32_t z_off0 = SLOT_W + SLOT_S + g8 * CW + warp;
    const uint32_t z_off1 = z_off0 + 8 * CW;
    float y[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) y[nb][i] = 0.0f;

    uint32_t slot = 0, phase = 0;
    for (int i = 0; ok && i < nstages; ++i) {
        const int j = i / KS, ks = i - j * KS;
        if (!warp_wait(&full[slot], phase, abort_flag, tmo, false)) {
            ok = false;
            break;
        }
        const uint32_t st = ring_base + slot * SLOT_BYTES;
        const uint4 w0 = lds128(st + w_off0);
        const uint4 w1 = lds128(st + w_off1);
        const uint32_t s0 = lds_u16(st + s_off0), s1 = lds_u16(st + s_off1);
        const uint32_t z0 = lds_u8(st + z_off0), z1 = lds_u8(st + z_off1);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (++slot == static_cast<uint32_t>(S)) {
            slot = 0;
            phase ^= 1u;
        }

        // B fragments of this group for my activation rows g8 (+ 8).
        const int g = ks * CW + warp;
        uint4 bf[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int m = g8 + 8 * nb;
#pragma unroll
            for (int v = 0; v < 4; ++v)
                bf[nb][v] = m < M ? lds128(a_base + ((((g * 4 + v) * M + m) * 4 + t4) << 4)) : make_uint4(0, 0, 0, 0);
        }

        const uint32_t zz0 = kBf16x2_128 + z0 * 0x00010001u;   // bf16 pair (128 + zp)
        const uint32_t zz1 = kBf16x2_128 + z1 * 0x00010001u;
        float d[NB][2][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) d[nb][h][e] = 0.0f;
        const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w};
        const uint32_t wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint32_t pa[4], pb[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                pa[k] = bsub2(level_pair(wa[v] >> (4 * k)), zz0);
                pb[k] = bsub2(level_pair(wb[v] >> (4 * k)), zz1);
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                mma_bf16(d[nb][0], pa[0], pb[0], pa[1], pb[1], bf[nb][v].x, bf[nb][v].y);
                mma_bf16(d[nb][1], pa[2], pb[2], pa[3], pb[3], bf[nb][v].z, bf[nb][v].w);
            }
        }
        const float sf0 = half_bits_to_f32(s0), sf1 = half_bits_to_f32(s1);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            y[nb][0] = fmaf(sf0, __fadd_rn(d[nb][0][0], d[nb][1][0]), y[nb][0]);
            y[nb][1] = fmaf(sf0, __fadd_rn(d[nb][0][1], d[nb][1][1]), y[nb][1]);
            y[nb][2] = fmaf(sf1, __fadd_rn(d[nb][0][2], d[nb][1][2]), y[nb][2]);
            y[nb][3] = fmaf(sf1, __fadd_rn(d[nb][0][3], d[nb][1][3]), y[nb][3]);
        }

        if (ks == KS - 1) {  // tile done: partial sums to the reduction area
            const int b = j & 1;
            if (!warp_wait(&red_empty[b], static_cast<uint32_t>(((j >> 1) & 1) ^ 1), abort_flag, tmo, false)) {
                ok = false;
                break;
            }
            float *rb = red + (b * CW + warp) * COLS * RED_STRIDE;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int c = 8 * nb + 2 * t4;
                rb[c * RED_STRIDE + g8] = y[nb][0];
                rb[(c + 1) * RED_STRIDE + g8] = y[nb][1];
                rb[c * RED_STRIDE + g8 + 8] = y[nb][2];
                rb[(c + 1) * RED_STRIDE + g8 + 8] = y[nb][3];
#pragma unroll
                for (int e = 0; e < 4; ++e) y[nb][e] = 0.0f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&red_full[b]);
        }
    }
}

// Tensor maps of one launch: qweight as (64 B, row, group) with box (64, 16, 16); scales
// and zero points as [row][group] with box (16 groups, 16 rows).  Strides are multiples
// of 16 bytes when K is a multiple of 2048 and the bases are 16-byte aligned.
inline bool make_maps(CUtensorMap *tmW, CUtensorMap *tmS, CUtensorMap *tmZ, const uint8_t *qweight,
                      const __half *scales, const uint8_t *zeros, int64_t N, int64_t K) {
    auto fn = gemm::encode_fn();
    if (!fn) return false;
    const uint64_t ng = static_cast<uint64_t>(K / 128);
    const cuuint64_t wd[3] = {GROUP_BYTES, static_cast<cuuint64_t>(N), ng};
    const cuuint64_t ws[2] = {static_cast<cuuint64_t>(K / 2), GROUP_BYTES};
    const cuuint32_t wb[3] = {GROUP_BYTES, ROWS, CW};
    const cuuint32_t es[3] = {1, 1, 1};
    if (fn(tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(qweight), wd, ws, wb, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    return gemm::make_map_2d(tmS, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, ng, N, ng * 2, CW, ROWS,
                             CU_TENSOR_MAP_SWIZZLE_NONE) &&
           gemm::make_map_2d(tmZ, CU_TENSOR_MAP_DATA_TYPE_UINT8, zeros, ng, N, ng, CW, ROWS,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace gmma
}  // namespace w4
