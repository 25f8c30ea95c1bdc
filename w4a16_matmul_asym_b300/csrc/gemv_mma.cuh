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
// CTA per SM).  A stage is one tile's k-slice of 16 * GPW groups (GPW = 2 when K is a
// multiple of 4096, else 1), brought in by three tensor copies that complete on the
// stage's mbarrier: the packed levels through a 3-D tensor map that views qweight as
// (128 bytes = 2 groups, row, group pair), box (128, 16, 8 GPW), with 128-byte swizzle,
// so they land as [pair][row][128 B] with the 16-byte chunk c of row r stored at
// c ^ (r & 7); the scales and zero points through 2-D maps.  Rows past N are
// zero-filled by the copy.  Up to MAX_STAGES stages are in flight.  When a tile is a
// single stage and M <= 8, warp w uses the same groups of A in every tile, so each lane
// loads its B fragments once, straight from global memory into registers (RB).
// Otherwise the activations are copied once per CTA into shared memory, permuted so
// that every B fragment is one conflict-free 16-byte load.  Int8 activations (W4A8) are
// widened to bf16 on the way, exactly, since |a_q| <= 128.
//
// Bank conflicts.  The 8 lanes of a quarter warp read MMA rows g and g + 1 (4 chunks
// each).  MMA row g reads physical row pi(g) = (g >> 1) + 4 (g & 1) of the tile (and
// g + 8 reads pi(g) + 8), so the two rows of a quarter warp differ in bit 2 and their
// swizzled chunks fall in opposite halves of the 128-byte bank window.  The output of
// MMA row g is written back as row pi(g).
//
// Work split.  Consumer warp w takes quantization groups w + 16 j (j < GPW) of every
// stage, i.e. split-K across the 16 warps, with GPW independent dependency chains per
// warp to hide the latency of shared-memory loads and MMAs; its partial sums of a tile
// stay in registers across the tile's stages and go to a double-buffered reduction
// area at the tile's end; an epilogue warp adds the 16 partials in a fixed order
// (deterministic), applies the optional per-row factor (the W4A8 activation scale),
// rounds to bf16 and stores Y.
//
// Launch: with programmatic dependent launch, so the next kernel's launch overlaps this
// one's tail; every thread waits (griddepcontrol.wait) for the preceding kernel in the
// stream before reading global memory.  Only an L2 prefetch of the first 64 KB of the
// CTA's weight band goes out earlier (prefetch.cuh: a hint that reads nothing into the CTA);
// it measured 3-6 % faster on every decode shape tried, e.g. 5.49 -> 5.24 us for M = 8,
// N = K = 4096 and 31.1 -> 30.4 us for M = 8, 28672 x 8192.
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
#include "prefetch.cuh"
#include "gemm_tcgen05.cuh"   // tensor-map encoding (driver entry point)

namespace w4 {
namespace gmma {

constexpr int CW = 16;                        // consumer warps
constexpr int PRODUCER = CW;                  // warp index of the producer
constexpr int EPILOGUE = CW + 1;              // warp index of the epilogue
constexpr int NUM_THREADS = (CW + 2) * 32;
constexpr int ROWS = 16;                      // W rows per tile (the MMA's M)
constexpr int PAIR_BYTES = 128;               // packed bytes of two groups of one row
constexpr int MAX_STAGES = 12;
constexpr int RED_STRIDE = 20;                // floats per (warp, column): conflict-free writes
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr uint32_t kBf16x2_128 = 0x43004300u;  // bf16 pair (128, 128)

// Stage geometry for GPW groups per warp per stage.
__host__ __device__ constexpr int groups_per_stage(int gpw) { return CW * gpw; }
__host__ __device__ constexpr int k_per_stage(int gpw) { return 128 * CW * gpw; }
__host__ __device__ constexpr int slot_w(int gpw) { return ROWS * 64 * CW * gpw; }   // [pair][row][128 B]
__host__ __device__ constexpr int slot_s(int gpw) { return ROWS * CW * gpw * 2; }    // fp16 [row][group]
__host__ __device__ constexpr int slot_z(int gpw) { return ROWS * CW * gpw; }        // uint8 [row][group]
__host__ __device__ constexpr int slot_sz(int gpw) { return slot_s(gpw) + slot_z(gpw); }
__host__ __device__ constexpr int slot_bytes(int gpw) { return slot_w(gpw) + slot_sz(gpw); }

__host__ __device__ constexpr int red_bytes(int nb) { return 2 * CW * 8 * nb * RED_STRIDE * 4; }
__host__ __device__ constexpr int a_bytes(int M, int K) { return (M * K * 2 + 1023) / 1024 * 1024; }
__host__ __device__ constexpr int bar_bytes() { return (2 * MAX_STAGES + 5) * 8 + 16; }
// Layout (offsets from a 1024-byte aligned base): activations (bf16, permuted), the W
// parts of every stage (1024-byte aligned for the swizzle), their scale/zero parts, the
// reduction area, the barriers; plus 1024 bytes of slack for aligning the base.
__host__ __device__ constexpr int smem_bytes(int M, int K, int nb, int gpw, int stages, bool regb = false) {
    return 1024 + (regb ? 0 : a_bytes(M, K)) + stages * slot_bytes(gpw) + red_bytes(nb) + bar_bytes();
}
// Whether the activations can stay in registers: one 8-column block and one stage per
// tile (K = 2048 GPW), so every warp uses the same GPW groups of A in every tile.
__host__ __device__ constexpr bool regb_ok(int M, int K, int gpw) { return M <= 8 && K == k_per_stage(gpw); }
// MMA row g (0..7) reads physical tile row pi(g); rows g + 8 read pi(g) + 8.
__host__ __device__ constexpr int row_of(int g) { return (g >> 1) + 4 * (g & 1); }

struct Params {
    const void *A;            // [M, K]: bf16 activations, or int8 ones (W4A8)
    const uint8_t *qweight;   // [N, K/2]
    const __half *scales;     // [N, K/128]
    const uint8_t *zeros;     // [N, K/128]
    const float *row_scale;   // [M] factor applied to each output row before rounding, or null
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
// 8 consecutive int8 (natural order) -> the same (k, k+4) bf16 pairs, exactly.
__device__ __forceinline__ uint32_t bf16x2_of_i8(uint32_t lo_byte, uint32_t hi_byte) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(static_cast<float>(static_cast<int8_t>(lo_byte & 0xFFu)),
                                                   static_cast<float>(static_cast<int8_t>(hi_byte & 0xFFu)));
    return *reinterpret_cast<const uint32_t *>(&b);
}
__device__ __forceinline__ uint4 pair_permute_i8(uint2 nat) {
    uint4 r;
    r.x = bf16x2_of_i8(nat.x, nat.y);              // a0, a4
    r.y = bf16x2_of_i8(nat.x >> 8, nat.y >> 8);    // a1, a5
    r.z = bf16x2_of_i8(nat.x >> 16, nat.y >> 16);  // a2, a6
    r.w = bf16x2_of_i8(nat.x >> 24, nat.y >> 24);  // a3, a7
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
// The whole warp waits (common.cuh: every lane polls, a vote decides).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned long long tmo, bool polite) {
    return warp_mbar_wait(bar, parity, abort_flag, tmo, polite);
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

// One thread issues every stage: three tensor copies (x coordinates 0 and 16 GPW ks,
// both multiples of 16 bytes).
template <int GPW>
__device__ __forceinline__ void produce(const Params &p, const CUtensorMap *tmW, const CUtensorMap *tmS,
                                        const CUtensorMap *tmZ, uint8_t *ring_w, uint8_t *ring_sz, uint64_t *full,
                                        uint64_t *empty, volatile int *abort_flag, int t_begin, int nstages) {
    if (lane_id() != 0) return;
    constexpr int GPS = groups_per_stage(GPW);
    const int KS = p.K / k_per_stage(GPW), S = p.stages;
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
        uint8_t *sz = ring_sz + static_cast<size_t>(slot) * slot_sz(GPW);
        mbar_arrive_expect_tx(&full[slot], slot_bytes(GPW));
        tma_load_3d(ring_w + static_cast<size_t>(slot) * slot_w(GPW), tmW, &full[slot], 0, n0, ks * (GPS / 2), pol);
        tma_load_2d(sz, tmS, &full[slot], ks * GPS, n0, pol);
        tma_load_2d(sz + slot_s(GPW), tmZ, &full[slot], ks * GPS, n0, pol);
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
    float rs[COLS / 2];
#pragma unroll
    for (int i = 0; i < COLS / 2; ++i) {
        const int m = (lane >> 4) + 2 * i;
        rs[i] = (p.row_scale != nullptr && m < p.M) ? p.row_scale[m] : 1.0f;
    }
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
                if (m < p.M) p.Y[static_cast<int64_t>(m) * p.N + n] = __float2bfloat16_rn(__fmul_rn(acc[i], rs[i]));
            }
        }
    }
}

// ---- the kernel ----------------------------------------------------------------------------
// NB = number of 8-column activation blocks (1: M <= 8, 2: M <= 16); GPW = groups per
// warp per stage; I8 = int8 activations (widened to bf16 while staged); RB = activations
// held in registers instead of shared memory (only when regb_ok: NB = 1, one stage per tile).
template <int NB, int GPW, bool I8, bool RB>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmZ, const Params p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // The 128-byte swizzle of the W copies assumes 1024-byte aligned shared offsets.
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    constexpr int COLS = 8 * NB;
    constexpr int GPS = groups_per_stage(GPW);
    constexpr int SW = slot_w(GPW), SSZ = slot_sz(GPW), SS = slot_s(GPW);
    const int M = p.M, K = p.K;
    const int KS = K / k_per_stage(GPW);
    const int S = p.stages;
    static_assert(!RB || NB == 1, "register-held activations take one 8-column block");
    uint8_t *ring_w = smem + (RB ? 0 : a_bytes(M, K));
    uint8_t *ring_sz = ring_w + static_cast<size_t>(S) * SW;
    float *red = reinterpret_cast<float *>(ring_sz + static_cast<size_t>(S) * SSZ);
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
    // The band's first 64 KB of weights start towards L2 while the preceding kernel drains
    // (a hint: nothing is read into the CTA before the wait).
    if (warp == PRODUCER && lane == 0)
        prefetch_weight_band_l2(p.qweight, p.scales, p.zeros, static_cast<int64_t>(t_begin) * ROWS,
                                min(static_cast<int64_t>(t_end) * ROWS, static_cast<int64_t>(p.N)), K, 65536);
    pdl_wait_then_release();   // no global memory is read into the CTA before this point

    if (warp == PRODUCER) {
        produce<GPW>(p, &tmW, &tmS, &tmZ, ring_w, ring_sz, full, empty, abort_flag, t_begin, nstages);
        return;
    }
    if (warp == EPILOGUE) {
        epilogue<NB>(p, red, red_full, red_empty, abort_flag, t_begin, ntiles);
        return;
    }

    const int g8 = lane >> 2, t4 = lane & 3;
    // ---- consumers, RB: with one stage per tile, warp w uses groups w + 16 h of A in
    // every tile, so lane (g8, t4) loads its B fragments once: A[g8, 128 (w + 16 h) + 32 t4
    // + 8 v + (0 4 1 5 2 6 3 7)] for v < 4 (64 contiguous bytes of row g8 per group,
    // permuted in registers).  Rows g8 >= M are zero.  No shared memory, no barrier.
    uint4 breg[RB ? GPW : 1][4];
    if constexpr (RB) {
#pragma unroll
        for (int h = 0; h < GPW; ++h) {
            const int64_t e0 = static_cast<int64_t>(g8) * K + 128 * (warp + CW * h) + 32 * t4;
            uint4 nat[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                nat[v] = make_uint4(0, 0, 0, 0);
                if (g8 < M) {
                    if constexpr (I8) {
                        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(static_cast<const int8_t *>(p.A) + e0 + 8 * v));
                        nat[v] = make_uint4(q.x, q.y, 0, 0);
                    } else {
                        nat[v] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.A) + e0 + 8 * v));
                    }
                }
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                if constexpr (I8) breg[h][v] = g8 < M ? pair_permute_i8(make_uint2(nat[v].x, nat[v].y)) : nat[v];
                else breg[h][v] = pair_permute(nat[v]);
            }
        }
    }
    // ---- consumers: stage the activations, permuted: the 16-byte chunk (g, v, m, t)
    // (index ((4 g + v) M + m) 4 + t) holds A[m, 128 g + 32 t + 8 v + (0 4 1 5 2 6 3 7)]
    // as bf16.  Threads walk A in its natural order, so each warp's loads are contiguous
    // (coalesced), and scatter the permuted chunks into shared memory.
    const uint32_t a_base = smem_addr(smem);
    if constexpr (!RB) {
        const int total = M * (K >> 3);
        constexpr int BATCH = 8;
        for (int c0 = threadIdx.x; c0 < total; c0 += BATCH * CW * 32) {
            uint4 nat[BATCH];
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int c = c0 + u * CW * 32;
                nat[u] = make_uint4(0, 0, 0, 0);
                if (c < total) {
                    const int64_t e = static_cast<int64_t>(c) * 8;
                    if constexpr (I8) {
                        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(static_cast<const int8_t *>(p.A) + e));
                        nat[u] = make_uint4(q.x, q.y, 0, 0);
                    } else {
                        nat[u] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.A) + e));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int c = c0 + u * CW * 32;
                if (c < total) {
                    uint4 v;
                    if constexpr (I8) v = pair_permute_i8(make_uint2(nat[u].x, nat[u].y));
                    else v = pair_permute(nat[u]);
                    const int m = c / (K >> 3), kc = c - m * (K >> 3);
                    const int g = kc >> 4, t = (kc >> 2) & 3, vv = kc & 3;
                    const int d = (((4 * g + vv) * M + m) << 2) + t;
                    sts128(a_base + (static_cast<uint32_t>(d) << 4), v);
                }
            }
        }
    }
    if constexpr (!RB) named_barrier_sync(1, CW * 32);

    bool ok = true;
    if (p.wait.stall) ok = warp_wait(never, 0, abort_flag, tmo, false);  // test hook

    const int r0 = row_of(g8), r1 = r0 + 8;        // physical rows of MMA rows g8, g8 + 8
    const uint32_t ringw_base = smem_addr(ring_w), ringsz_base = smem_addr(ring_sz);
    // Group w + 16 j of a stage sits in pair (w >> 1) + 8 j, half w & 1: its 16-byte chunk
    // c = 4 (w & 1) + t4, swizzled by r & 7 (the same for r0 and r1).
    const uint32_t chunk = static_cast<uint32_t>(((warp & 1) * 4 + t4) ^ (r0 & 7)) << 4;
    const uint32_t w_off0 = (warp >> 1) * (ROWS * PAIR_BYTES) + r0 * PAIR_BYTES + chunk;
    constexpr uint32_t W_J = 8 * ROWS * PAIR_BYTES;   // offset of group w + 16 from group w
    // Scale / zero-point offsets within a stage, and the B-fragment addresses: chunk
    // ((4 g + v) M + m) 4 + t with g = GPS ks + warp + 16 h, so every address is a fixed
    // per-lane base plus (ks, h, v, nb) multiples of compile-time or loop-invariant strides.
    const uint32_t s_off0 = r0 * (GPS * 2) + warp * 2, s_off1 = r1 * (GPS * 2) + warp * 2;
    const uint32_t z_off0 = SS + r0 * GPS + warp, z_off1 = SS + r1 * GPS + warp;
    const uint32_t b_row = 64u * M;                        // bytes from (g, v) to (g, v + 1)
    const uint32_t b_lane = a_base + ((warp * 4 * M + g8) * 4 + t4) * 16;
    const uint32_t b_stage = b_row * 4 * GPS;              // bytes per stage of groups
    bool bvalid[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) bvalid[nb] = g8 + 8 * nb < M;
    float y[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) y[nb][i] = 0.0f;

    uint32_t slot = 0, phase = 0;
    int j = 0, ks = 0;                                     // tile within the CTA, stage within the tile
    uint32_t b_ks = b_lane;
    for (int i = 0; ok && i < nstages; ++i) {
        if (!warp_wait(&full[slot], phase, abort_flag, tmo, false)) {
            ok = false;
            break;
        }
        const uint32_t stw = ringw_base + slot * SW, stsz = ringsz_base + slot * SSZ;
        uint32_t wa[GPW][4], wb[GPW][4], zz0[GPW], zz1[GPW];
        float sf0[GPW], sf1[GPW];
#pragma unroll
        for (int h = 0; h < GPW; ++h) {
            const uint4 w0 = lds128(stw + w_off0 + h * W_J);
            const uint4 w1 = lds128(stw + w_off0 + h * W_J + 8 * PAIR_BYTES);
            wa[h][0] = w0.x; wa[h][1] = w0.y; wa[h][2] = w0.z; wa[h][3] = w0.w;
            wb[h][0] = w1.x; wb[h][1] = w1.y; wb[h][2] = w1.z; wb[h][3] = w1.w;
            sf0[h] = half_bits_to_f32(lds_u16(stsz + s_off0 + h * (CW * 2)));
            sf1[h] = half_bits_to_f32(lds_u16(stsz + s_off1 + h * (CW * 2)));
            zz0[h] = kBf16x2_128 + lds_u8(stsz + z_off0 + h * CW) * 0x00010001u;  // bf16 pair (128 + zp)
            zz1[h] = kBf16x2_128 + lds_u8(stsz + z_off1 + h * CW) * 0x00010001u;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (++slot == static_cast<uint32_t>(S)) {
            slot = 0;
            phase ^= 1u;
        }

        float d[GPW][NB][2][4];
#pragma unroll
        for (int h = 0; h < GPW; ++h)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int e = 0; e < 4; ++e) d[h][nb][q][e] = 0.0f;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
#pragma unroll
            for (int h = 0; h < GPW; ++h) {
                uint32_t pa[4], pb[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    pa[k] = bsub2(level_pair(wa[h][v] >> (4 * k)), zz0[h]);
                    pb[k] = bsub2(level_pair(wb[h][v] >> (4 * k)), zz1[h]);
                }
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    // group GPS ks + warp + 16 h, piece v, activation row g8 + 8 nb
                    uint4 bf;
                    if constexpr (RB) bf = breg[h][v];
                    else bf = bvalid[nb] ? lds128(b_ks + (CW * h * 4 + v) * b_row + nb * 512) : make_uint4(0, 0, 0, 0);
                    mma_bf16(d[h][nb][0], pa[0], pb[0], pa[1], pb[1], bf.x, bf.y);
                    mma_bf16(d[h][nb][1], pa[2], pb[2], pa[3], pb[3], bf.z, bf.w);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < GPW; ++h)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                y[nb][0] = fmaf(sf0[h], __fadd_rn(d[h][nb][0][0], d[h][nb][1][0]), y[nb][0]);
                y[nb][1] = fmaf(sf0[h], __fadd_rn(d[h][nb][0][1], d[h][nb][1][1]), y[nb][1]);
                y[nb][2] = fmaf(sf1[h], __fadd_rn(d[h][nb][0][2], d[h][nb][1][2]), y[nb][2]);
                y[nb][3] = fmaf(sf1[h], __fadd_rn(d[h][nb][0][3], d[h][nb][1][3]), y[nb][3]);
            }

        b_ks += b_stage;
        if (++ks == KS) {  // tile done: partial sums to the reduction area
            ks = 0;
            b_ks = b_lane;
            const int b = j & 1;
            if (!warp_wait(&red_empty[b], static_cast<uint32_t>(((j >> 1) & 1) ^ 1), abort_flag, tmo, false)) {
                ok = false;
                break;
            }
            float *rb = red + (b * CW + warp) * COLS * RED_STRIDE;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int c = 8 * nb + 2 * t4;
                rb[c * RED_STRIDE + r0] = y[nb][0];
                rb[(c + 1) * RED_STRIDE + r0] = y[nb][1];
                rb[c * RED_STRIDE + r1] = y[nb][2];
                rb[(c + 1) * RED_STRIDE + r1] = y[nb][3];
#pragma unroll
                for (int e = 0; e < 4; ++e) y[nb][e] = 0.0f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&red_full[b]);
            ++j;
        }
    }
}

// Tensor maps of one launch: qweight as (128 B, row, group pair) with box (128, 16, 8 GPW)
// and 128-byte swizzle; scales and zero points as [row][group] with box (16 GPW groups,
// 16 rows).  Strides are multiples of 16 bytes when K is a multiple of 2048 and the bases
// are 16-byte aligned.
inline bool make_maps(CUtensorMap *tmW, CUtensorMap *tmS, CUtensorMap *tmZ, const uint8_t *qweight,
                      const __half *scales, const uint8_t *zeros, int64_t N, int64_t K, int gpw) {
    auto fn = gemm::encode_fn();
    if (!fn) return false;
    const uint64_t ng = static_cast<uint64_t>(K / 128);
    const cuuint64_t wd[3] = {PAIR_BYTES, static_cast<cuuint64_t>(N), ng / 2};
    const cuuint64_t ws[2] = {static_cast<cuuint64_t>(K / 2), PAIR_BYTES};
    const cuuint32_t wb[3] = {PAIR_BYTES, ROWS, static_cast<cuuint32_t>(8 * gpw)};
    const cuuint32_t es[3] = {1, 1, 1};
    if (fn(tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(qweight), wd, ws, wb, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    const uint32_t gps = static_cast<uint32_t>(groups_per_stage(gpw));
    return gemm::make_map_2d(tmS, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, ng, N, ng * 2, gps, ROWS,
                             CU_TENSOR_MAP_SWIZZLE_NONE) &&
           gemm::make_map_2d(tmZ, CU_TENSOR_MAP_DATA_TYPE_UINT8, zeros, ng, N, ng, gps, ROWS,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Groups per warp per stage and ring depth for a shape, or 0 stages if it does not fit.
// The ring keeps about 64 KB of packed weights in flight per SM (2 stages of 32 KB, or 4
// of 16 KB), which covers an SM's share of the HBM bandwidth-latency product; deeper
// rings only delay each CTA's first stage.  Measured against the deepest ring that fits
// (4-5 stages of 32 KB): 9.13 -> 8.56 us at M = 8, 11008 x 4096; 11.07 -> 9.99 us at M = 4,
// 14336 x 4096; 16.98 -> 16.38 us at M = 8, 28672 x 4096; unchanged at 4096 x 4096 and
// 28672 x 8192.
inline void plan(int M, int K, int *gpw, int *stages) {
    const int nb = M <= 8 ? 1 : 2;
    *gpw = (nb == 1 && K % k_per_stage(2) == 0) ? 2 : 1;
    const int depth = 65536 / slot_w(*gpw) > 2 ? 65536 / slot_w(*gpw) : 2;
    *stages = 0;
    for (int s = depth < MAX_STAGES ? depth : MAX_STAGES; s >= 2; --s)
        if (smem_bytes(M, K, nb, *gpw, s) <= SMEM_LIMIT) {
            *stages = s;
            return;
        }
}

}  // namespace gmma
}  // namespace w4
