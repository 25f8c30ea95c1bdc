// gemm_tcgen05.cuh -- prefill-shaped W4A16 GEMM (M >= 9) on the 5th-generation
// tensor cores: Y[M,N] = A[M,K] * W_hat[N,K]^T, W_hat = (q - zp) * s16.
//
// The contraction is the fused dequantize-matmul of "Build a GPTQ INT4 Quantization
// Engine in Python/NumPy" (Step 5) with the dequantization of "From Scratch: Building a
// GPTQ INT4 Quantizer in Pure Python" (Step 4); "Building a From-Scratch Group-Wise INT4
// Quantization Layer for LLaMA Weights" (Architecture Overview) names fused
// dequant + matmul as the hot path.  The full-precision W never exists in memory:
// each 128 x 64 tile of packed W is dequantized to bf16 straight into tensor memory.
//
// The kernel computes the transposed product Y^T = W_hat * A^T so that the
// dequantized weights are the MMA's A operand, which tcgen05.mma reads from tensor
// memory (TMEM): MMA M = 128 rows of W, MMA N = MT rows of A (16..256, multiple of
// 16), K = 16 per instruction.  The activations are the B operand, loaded by TMA into
// 128-byte-swizzled shared memory.  Dequantized weights never touch shared memory,
// and every dequantized weight serves MT activation rows.
//
// One persistent CTA per SM, 640 threads (20 warps):
//   warp 0        TMA producer of the activation tiles [MT x 64] bf16
//   warp 1        allocates all 512 TMEM columns and runs the MMA loop; one elected
//                 lane issues the MMAs and their commits
//   warp 2        TMA producer of the packed W tiles, one quantization group (two
//                 k-blocks, [128 x 64 B], 64-byte swizzle) per copy, on a ring of its
//                 own so that dequantization runs ahead of the MMAs, bounded only by the
//                 TMEM A stages, and its latency stays off the MMAs' path.  A whole group
//                 per copy halves the copies' row requests; the swizzle spreads the
//                 dequantize threads' 16-byte reads (row pitch 64 B) over all banks
//   warps 4-11    epilogue: two warps per TMEM lane quarter, each draining half of the
//                 accumulator columns, 32 at a time, to bf16.  The accumulator is handed
//                 back to the MMA warp as soon as the last column is in registers; the
//                 values go through a per-warp shared-memory block [m][32 n] and one TMA
//                 tensor store per warp and tile, which runs under the next tile's MMAs
//                 (direct 2-byte stores instead when Y's rows are not 16-byte aligned)
//   warps 12-19   dequantize: two warps per lane quarter; thread = one row of the W
//                 tile, 32 of its 64 k of each k-block, one quantization group (one W
//                 stage, two k-blocks) per iteration -> tcgen05.st into two TMEM A stages
// TMEM: columns [0, 256) accumulators (two of 128 when MT <= 128, one of 256 otherwise),
// columns [256, 512) eight A-operand stages of 32 columns (64 bf16 per lane).
// Shared memory: 4 activation stages (32 KB), 4 packed-W stages (8 KB), then the
// epilogue's 8 x 8 KB store-staging blocks.
// Every wait is bounded (see common.cuh); on a timeout the CTA drains its copies and
// MMAs, frees TMEM and exits, leaving W4_ERR_TIMEOUT in the device error word.
#pragma once

#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"

namespace w4 {
namespace gemm {

constexpr int BW = 128;                       // W rows per tile (MMA M, TMEM lanes)
constexpr int BK = 64;                        // k per stage
constexpr int MT_MAX = 256;                   // activation rows per tile (MMA N), max
constexpr int SA = 4;                         // activation smem stages
constexpr int SW = 4;                         // packed-W smem stages (one quantization group each)
constexpr int ST = 8;                         // TMEM A-operand stages
constexpr int ACT_STAGE_MAX = MT_MAX * BK * 2;  // 32 KB
constexpr int BQ_STAGE = BW * BK;             // 8 KB: 128 rows x 64 B (two k-blocks)
constexpr int NUM_THREADS = 640;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int DEQ_WARP0 = 12;
constexpr int NUM_DEQ_WARPS = 8;
constexpr uint32_t BAR_EPI = 1;               // named barrier of the epilogue warps
constexpr uint32_t BAR_EPI_RS = 2;            // epilogue warps: the tile's row factors are staged
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;            // accumulator region
constexpr uint32_t A_COLS = 32;               // one A stage: 64 bf16 per lane
static_assert(ST % 2 == 0, "dequantize warps take TMEM A stages in pairs");

constexpr int Y_WARP_BYTES = (MT_MAX / 2) * 32 * 2;  // one epilogue warp's [m][32 n] bf16 block

constexpr int OFF_ACT = 0;
constexpr int OFF_W = OFF_ACT + SA * ACT_STAGE_MAX;
constexpr int OFF_YST = OFF_W + SW * BQ_STAGE;
constexpr int OFF_BAR = OFF_YST + NUM_EPI_WARPS * Y_WARP_BYTES;
constexpr int NUM_BARS = 2 * SA + 2 * SW + 2 * ST + 4 + 2;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
// The current tile's per-row factors (W4A8), fp32; 32 spare entries let a chunk of 32
// columns read past the tile's last column (those columns are never stored).
constexpr int RS_ENTRIES = MT_MAX + 32;
constexpr int OFF_RS = OFF_MISC + 16;
constexpr int SMEM_BYTES = OFF_RS + RS_ENTRIES * 4;
constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory per CTA");

// Instruction descriptor of tcgen05.mma.kind::f16: fp32 D, bf16 A and B, both
// K-major, N = mt, M = 128.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t mt) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((mt >> 3) << 17) |
           (static_cast<uint32_t>(BW >> 4) << 24);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) |
           (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Warp-wide forms: every lane of a converged warp executes them (so the operands stay
// warp-uniform) and elect.sync picks the one lane that issues, the same lane each time
// for a fully active warp, so its commits track its own MMAs.
__device__ __forceinline__ void umma_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit_warp(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_addr(bar))
        : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane <- registers.
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 8 consecutive 32-bit columns of this thread's TMEM lane -> registers.
__device__ __forceinline__ void tmem_ld_8cols(uint32_t taddr, uint32_t *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity,
                                                unsigned long long timeout_ns) {
    const uint32_t a = smem_addr(bar);
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(a, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) {
            record_error(W4_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// The whole warp waits (common.cuh: every lane polls, a vote decides).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned long long timeout_ns) {
    return warp_mbar_wait(bar, parity, abort_flag, timeout_ns);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;  // (a & b) | c
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 8 packed levels (element 2j low nibble) -> 4 words of bf16 pairs (q - zp) * s, in k
// order.  Each nibble pair is spread into the two halves of a word with prmt, masked
// and ORed with the bf16 pattern of 128 (ulp 1), giving 128 + q exactly; subtracting
// 128 + zp is exact; the multiply by the bf16 scale rounds once.
__device__ __forceinline__ void dequant8(uint32_t x, uint32_t zz2, uint32_t s2, uint32_t *o) {
    const uint32_t x4 = x >> 4;
    const uint32_t magic = 0x43004300u, mask = 0x000F000Fu;
    o[0] = bf16x2_mul(bf16x2_sub(lop3_and_or(prmt(x, x4, 0x0400u), mask, magic), zz2), s2);
    o[1] = bf16x2_mul(bf16x2_sub(lop3_and_or(prmt(x, x4, 0x0501u), mask, magic), zz2), s2);
    o[2] = bf16x2_mul(bf16x2_sub(lop3_and_or(prmt(x, x4, 0x0602u), mask, magic), zz2), s2);
    o[3] = bf16x2_mul(bf16x2_sub(lop3_and_or(prmt(x, x4, 0x0703u), mask, magic), zz2), s2);
}

__device__ __forceinline__ uint32_t bf16_bits(float f) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f)));
}

// One TMA producer thread: for each k-block of this CTA's tiles in order, waits for a
// free stage of its ring and copies one box into it (activations: [mt x 64] at
// (k, m), one per k-block; packed W: [128 x 64 B] at (k / 2, n), one per pair of
// k-blocks).  On an abort it waits for every copy it issued to land before returning.
template <int S, bool kW>
__device__ __forceinline__ void produce(const CUtensorMap *map, uint8_t *ring, uint32_t stage_bytes,
                                        uint32_t tx_bytes, uint64_t *full, uint64_t *empty,
                                        int num_tiles, int m_tiles, int KB, int mt,
                                        volatile int *abort_flag, unsigned long long tmo) {
    const uint64_t pol = policy_evict_last();
    int issued_parity[S];
#pragma unroll
    for (int s = 0; s < S; ++s) issued_parity[s] = -1;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int mi = tile % m_tiles, ni = tile / m_tiles;
        for (int kb = 0; kb < KB; kb += (kW ? 2 : 1)) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, tmo)) {
                ok = false;
                break;
            }
            uint8_t *st = ring + stage * stage_bytes;
            mbar_arrive_expect_tx(&full[stage], tx_bytes);
            if (kW)
                tma_load_2d(st, map, &full[stage], kb * (BK / 2), ni * BW, pol);
            else
                tma_load_2d(st, map, &full[stage], kb * BK, mi * mt, pol);
#pragma unroll
            for (int s = 0; s < S; ++s)
                if (s == static_cast<int>(stage)) issued_parity[s] = static_cast<int>(phase);
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        // Drain: every copy this thread issued must land before the CTA exits.
#pragma unroll
        for (int s = 0; s < S; ++s)
            if (issued_parity[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(issued_parity[s]), tmo);
    }
}

// Named barrier over `threads` (whole warps) that also ORs one flag from every thread,
// so that all participants take the same decision.
__device__ __forceinline__ uint32_t named_bar_or(uint32_t id, uint32_t threads, uint32_t flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %3, 0;\n\t"
        "bar.red.or.pred q, %1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(threads), "r"(flag)
        : "memory");
    return r;
}

struct Params {
    const __half *scales;
    const uint8_t *zeros;
    __nv_bfloat16 *Y;
    const float *row_scale;  // optional per-activation-row factor applied before rounding (W4A8)
    int M, N, K;
    int mt;          // activation rows per tile (MMA N): multiple of 16, <= 256
    uint32_t idesc;  // instruction descriptor for (M = 128, N = mt)
    int tma_store;   // 1: Y written by TMA tensor stores (tmY valid), 0: direct stores
    WaitParams wait;
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmY, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    // Align the shared-window offset (not the generic address) to 1024 bytes, as the
    // 128-byte swizzle pattern of TMA and of the MMA descriptors assumes.
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *act_full = bars;           // activation tile landed (TMA)
    uint64_t *act_empty = act_full + SA;  // activation stage consumed (MMA commit)
    uint64_t *w_full = act_empty + SA;    // packed W tile landed (TMA)
    uint64_t *w_empty = w_full + SW;      // packed W stage read (dequant warps)
    uint64_t *a_full = w_empty + SW;      // TMEM A stage written (dequant warps)
    uint64_t *a_empty = a_full + ST;    // TMEM A stage consumed (MMA commit)
    uint64_t *acc_full = a_empty + ST;  // accumulator complete (MMA commit)
    uint64_t *acc_empty = acc_full + 2;  // accumulator drained (epilogue warps)
    uint64_t *mma_done = acc_empty + 2;
    uint64_t *never = mma_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int mt = p.mt;
    const int m_tiles = (p.M + mt - 1) / mt;
    const int n_tiles = (p.N + BW - 1) / BW;
    const int num_tiles = m_tiles * n_tiles;
    const int KB = p.K / BK;
    const int num_acc = (mt <= 128) ? 2 : 1;
    const unsigned long long tmo = p.wait.timeout_ns;
    const int act_bytes = mt * BK * 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(&act_full[s], 1);
            mbar_init(&act_empty[s], 1);
        }
        for (int s = 0; s < SW; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], NUM_DEQ_WARPS);
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(&a_full[s], NUM_DEQ_WARPS);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], NUM_EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.tma_store) prefetch_tensormap(&tmY);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer: activations ----------------
        if (lane == 0)
            produce<SA, false>(&tmA, smem + OFF_ACT, ACT_STAGE_MAX, static_cast<uint32_t>(act_bytes),
                               act_full, act_empty, num_tiles, m_tiles, KB, mt, abort_flag, tmo);
        __syncwarp();
    } else if (warp == 2) {
        // ---------------- TMA producer: packed W ----------------
        if (lane == 0)
            produce<SW, true>(&tmB, smem + OFF_W, BQ_STAGE, BQ_STAGE, w_full, w_empty, num_tiles, m_tiles,
                              KB, mt, abort_flag, tmo);
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // The whole warp runs the loop; one elected lane issues the MMAs and commits.
        uint32_t stage = 0, phase = 0, as = 0, aphase = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        if (p.wait.stall) ok = warp_wait(never, 0, abort_flag, tmo);  // test hook
        // Descriptor of activation stage 0; the start address field (bytes / 16) moves by
        // ACT_STAGE_MAX / 16 per stage and by 2 per 16-k step.
        const uint64_t bdesc0 = sw128_desc(smem_addr(smem + OFF_ACT));
        const uint32_t idesc = p.idesc;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            if (!warp_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, tmo)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * 128u;
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait(&act_full[stage], phase, abort_flag, tmo) ||
                    !warp_wait(&a_full[as], aphase, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(stage * (ACT_STAGE_MAX >> 4));
                const uint32_t a_tmem = tmem_base + ACC_COLS + as * A_COLS;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    umma_tmem_a_warp(d_tmem, a_tmem + kk * 8, bdesc + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
                umma_commit_warp(&act_empty[stage]);
                umma_commit_warp(&a_empty[as]);
                if (++stage == SA) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++as == ST) {
                    as = 0;
                    aphase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit_warp(&acc_full[acc]);
            if (++acc == static_cast<uint32_t>(num_acc)) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // All MMAs issued by the elected lane complete before TMEM is released.
        umma_commit_warp(mma_done);
        if (lane == 0) mbar_wait_drain(mma_done, 0, tmo);
        __syncwarp();
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + NUM_EPI_WARPS) {
        // ---------------- epilogue: TMEM -> bf16 -> Y ----------------
        const int quarter = warp & 3;                  // TMEM lanes [32q, 32q + 32)
        const int half = (warp - EPI_WARP0) >> 2;      // which half of the tile's columns
        const int cols = mt >> 1;                      // columns per half (multiple of 8)
        // This warp's staging block: `cols` rows of m, 32 consecutive n (64 bytes) each.
        unsigned short *ystage =
            reinterpret_cast<unsigned short *>(smem + OFF_YST + (warp - EPI_WARP0) * Y_WARP_BYTES);
        float *rs_s = reinterpret_cast<float *>(smem + OFF_RS);
        const int et = (warp - EPI_WARP0) * 32 + lane;    // 0 .. 255: one tile row factor each
        uint32_t acc = 0, acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int mi = tile % m_tiles, ni = tile / m_tiles;
            // The row factors of the tile's activation rows, one per epilogue thread,
            // loaded before the accumulator wait so that their latency hides under it.
            float my_rs = 1.0f;
            if (p.row_scale != nullptr && et < mt) {
                const int mr = mi * mt + et;
                my_rs = __ldg(p.row_scale + (mr < p.M ? mr : p.M - 1));
            }
            // One warp polls the accumulator barrier; the others sleep on a named barrier
            // and leave the issue slots to the dequantize warps.  The OR of the poller's
            // result gives every warp the same decision.
            uint32_t stop = 0;
            if (warp == EPI_WARP0) stop = warp_wait(&acc_full[acc], acc_phase, abort_flag, tmo) ? 0u : 1u;
            if (named_bar_or(BAR_EPI, NUM_EPI_WARPS * 32, stop)) break;
            if (p.row_scale != nullptr) {
                // Every epilogue warp is past the previous tile (barrier above), so the
                // staged factors can be replaced; the second barrier publishes them.
                if (et < mt) rs_s[et] = my_rs;
                asm volatile("bar.sync %0, %1;" ::"n"(BAR_EPI_RS), "n"(NUM_EPI_WARPS * 32) : "memory");
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   acc * 128u + static_cast<uint32_t>(half * cols);
            const int n = ni * BW + quarter * 32 + lane;
            const int m0 = mi * mt + half * cols;
            unsigned short *y = reinterpret_cast<unsigned short *>(p.Y) + n;
            if (p.tma_store) {
                // The previous tile's store out of this block has finished reading it.
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
            }
#pragma unroll 1
            for (int c0 = 0; c0 < cols; c0 += 32) {
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (c0 + 8 * j < cols) tmem_ld_8cols(tbase + c0 + 8 * j, v + 8 * j);
                tmem_wait_ld();
                if (p.row_scale != nullptr) {
                    // Column j of this chunk is activation row m0 + c0 + j, tile row
                    // half * cols + c0 + j: scale it in fp32 by the staged factor (the same
                    // shared-memory word in every lane: a broadcast).  Loading the factors
                    // from global memory here, per chunk, cost 22 us on 2048 x 14336 x 4096.
                    const float *rsc = rs_s + half * cols + c0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__fmul_rn(__uint_as_float(v[j]), rsc[j]));
                }
                if (c0 + 32 >= cols) {
                    // This warp's part of the accumulator is in registers: hand it back.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[acc]);
                }
                if (p.tma_store) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < cols)
                            ystage[(c0 + j) * 32 + lane] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
                } else if (n < p.N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int m = m0 + c0 + j;
                        if (c0 + j < cols && m < p.M)
                            y[static_cast<int64_t>(m) * p.N] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
                    }
                }
            }
            if (p.tma_store) {
                // Generic-proxy writes of every lane before the async-proxy read of the store.
                fence_proxy_async_smem();
                __syncwarp();
                const int x = ni * BW + quarter * 32;
                if (lane == 0 && x < p.N && m0 < p.M) {
                    tma_store_2d(&tmY, ystage, x, m0);  // clipped at N and M
                    bulk_commit_group();
                }
                __syncwarp();
            }
            if (++acc == static_cast<uint32_t>(num_acc)) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // Stores issued by this warp complete before the CTA exits.
        if (p.tma_store && lane == 0) bulk_wait_group0();
        __syncwarp();
    } else if (warp >= DEQ_WARP0) {
        // ---------------- dequantize packed W -> TMEM A stages ----------------
        const int quarter = warp & 3;
        const int half = (warp - DEQ_WARP0) >> 2;      // which 32 of the 64 k of a stage
        const int r = quarter * 32 + lane;             // tile row owned by this thread
        const int ng = p.K / 128;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t ws = 0, wphase = 0, as = 0, aphase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            const int ni = tile / m_tiles;
            const int n = ni * BW + r;
            const bool valid = n < p.N;
            const int64_t sz_row = static_cast<int64_t>(n) * ng;
            // Scales / zero points run two groups ahead of use.
            uint32_t s_nx1 = 0, z_nx1 = 0, s_nx2 = 0, z_nx2 = 0;
            if (valid) {
                s_nx1 = __half_as_ushort(p.scales[sz_row]);
                z_nx1 = p.zeros[sz_row];
                if (ng > 1) {
                    s_nx2 = __half_as_ushort(p.scales[sz_row + 1]);
                    z_nx2 = p.zeros[sz_row + 1];
                }
            }
            // One quantization group (two k-blocks: W stages ws, ws + 1 and TMEM A stages
            // as, as + 1, both rings of even length) per iteration.
            for (int g = 0; g < ng; ++g) {
                const uint32_t s_cur = s_nx1, z_cur = z_nx1;
                s_nx1 = s_nx2;
                z_nx1 = z_nx2;
                if (valid && g + 2 < ng) {
                    s_nx2 = __half_as_ushort(p.scales[sz_row + g + 2]);
                    z_nx2 = p.zeros[sz_row + g + 2];
                }
                // bf16(s16) twice, and 128 + zp (exact) twice; invalid rows give 0.
                const uint32_t sb =
                    valid ? bf16_bits(__half2float(__ushort_as_half(static_cast<unsigned short>(s_cur))))
                          : 0u;
                const uint32_t zb = bf16_bits(128.0f + static_cast<float>(z_cur));
                const uint32_t s2 = sb | (sb << 16);
                const uint32_t zz2 = zb | (zb << 16);
                if (!warp_wait(&w_full[ws], wphase, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                const uint8_t *wrow = smem + OFF_W + ws * BQ_STAGE + r * 64;
                const int swz = (r >> 1) & 3;
                const uint4 w0 = *reinterpret_cast<const uint4 *>(wrow + 16 * (half ^ swz));
                const uint4 w1 = *reinterpret_cast<const uint4 *>(wrow + 16 * ((2 + half) ^ swz));
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[ws]);
                if (!warp_wait(&a_empty[as], aphase ^ 1u, abort_flag, tmo) ||
                    !warp_wait(&a_empty[as + 1], aphase ^ 1u, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = tmem_base + lane_addr + ACC_COLS + as * A_COLS + half * 16;
                uint32_t o[16];
                dequant8(w0.x, zz2, s2, o);
                dequant8(w0.y, zz2, s2, o + 4);
                dequant8(w0.z, zz2, s2, o + 8);
                dequant8(w0.w, zz2, s2, o + 12);
                tmem_st_16cols(dst, o);
                dequant8(w1.x, zz2, s2, o);
                dequant8(w1.y, zz2, s2, o + 4);
                dequant8(w1.z, zz2, s2, o + 8);
                dequant8(w1.w, zz2, s2, o + 12);
                tmem_st_16cols(dst + A_COLS, o);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_full[as]);
                    mbar_arrive(&a_full[as + 1]);
                }
                if (++ws == SW) {
                    ws = 0;
                    wphase ^= 1u;
                }
                if ((as += 2) == ST) {
                    as = 0;
                    aphase ^= 1u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---- host side ------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

inline bool make_map_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gemm

inline int launch_gemm_tcgen05(const __nv_bfloat16 *A, int64_t M, int64_t N, int64_t K,
                               const uint8_t *qweight, const __half *scales, const uint8_t *zeros,
                               __nv_bfloat16 *Y, cudaStream_t stream, int sms, WaitParams wp,
                               const float *row_scale = nullptr) {
    using namespace gemm;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return W4_ERR_UNSUPPORTED;
    const int mt = static_cast<int>(M >= MT_MAX ? MT_MAX : ((M + 15) / 16) * 16);
    CUtensorMap tmA, tmB;
    if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, K * 2, BK, mt,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return W4_ERR_CUDA;
    if (!make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qweight, K / 2, N, K / 2, BK, BW,
                     CU_TENSOR_MAP_SWIZZLE_64B))
        return W4_ERR_CUDA;
    // Y by tensor stores when its base and row pitch are 16-byte aligned: box of 32 n
    // (64 bytes) by mt / 2 rows of m, one per epilogue warp and tile.
    CUtensorMap tmY;
    memset(&tmY, 0, sizeof(tmY));
    const bool tma_store = (reinterpret_cast<uintptr_t>(Y) & 15u) == 0 && (N % 8) == 0;
    if (tma_store && !make_map_2d(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, N, M, N * 2, 32,
                                  static_cast<uint32_t>(mt / 2), CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4_ERR_CUDA;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4_ERR_CUDA;
    static std::once_flag attr_once[64];
    static cudaError_t attr_err[64];
    if (dev < 0 || dev >= 64) return W4_ERR_CUDA;
    std::call_once(attr_once[dev], [&]() {
        attr_err[dev] = cudaFuncSetAttribute(w4a16_gemm_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    });
    if (attr_err[dev] != cudaSuccess) return W4_ERR_CUDA;

    const int64_t tiles = ((M + mt - 1) / mt) * ((N + BW - 1) / BW);
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    Params prm;
    prm.scales = scales;
    prm.zeros = zeros;
    prm.Y = Y;
    prm.row_scale = row_scale;
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(N);
    prm.K = static_cast<int>(K);
    prm.mt = mt;
    prm.idesc = make_idesc(static_cast<uint32_t>(mt));
    prm.tma_store = tma_store ? 1 : 0;
    prm.wait = wp;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = stream;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, w4a16_gemm_kernel, tmA, tmB, tmY, prm);
    return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

}  // namespace w4
