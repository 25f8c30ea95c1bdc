// gemv_tc.cuh -- W4A16 matmul for a few activation rows (2 <= M <= 16) on the
// 5th-generation tensor cores.
//
// Computes Y[m,n] = sum_k A[m,k] * W_hat[n,k], W_hat = (q - zp) * s16, with fp32
// accumulation: the fused dequantize-matmul of "Build a GPTQ INT4 Quantization Engine
// in Python/NumPy" (Step 5) with the dequantization of "From Scratch: Building a GPTQ
// INT4 Quantizer in Pure Python" (Step 4), for batched decode.
//
// Why tensor cores here: the prefill GEMM tiles W by 128 rows, so for a small N it
// leaves most SMs idle.  This kernel splits K inside the MMA instead (below) and tiles
// W by 8 or 16 rows.  N carries all activation rows at once and the CUDA cores only
// unpack.  With a tile of only 8 or 16 rows, each tile's MMAs are short (four units of
// 64 levels for K = 4096) next to its fixed costs (the accumulator hand-off and an
// epilogue that reads one column per activation row and sums the parts), so the kernel
// runs well below both the MMA rate and HBM bandwidth; it is used for 9 <= M <= 16,
// where it beats the CUDA-core kernels, and not for M <= 8, where it does not.
//
// Layout of the contraction.  A tile is R = 128 / P rows of W, each split into P
// contiguous parts of KP = K / P levels; TMEM lane i holds row i / P, part i % P, so a
// tile is 8 or 16 rows and the rows spread evenly over all SMs for any N.  The MMA's B
// operand (N = MT * P rows, MT = M rounded up to keep N a multiple of 16) holds in row
// m * P + p the activations of row m in part p; D[i, m * P + p] is then the dot
// product of lane i's part with row m's activations in that part, and the epilogue
// reads, for every m, the column of its own part and sums the P parts of a row with
// xor shuffles.  The unpack warps write (q - zp) exactly (two levels per lop3 as bf16
// 128 + q, minus 128 + zp) and multiply by the group scale rounded to bf16 (one
// rounding, 2^-8 relative at most), as the prefill GEMM does.
//
// Order of levels inside the MMA K dimension (both operands use the same order):
//   * within a packed word (levels k0..k7) the bf16 pairs are (k_j, k_j+4), j = 0..3;
//   * within each 128-byte window of a part (8 chunks of 32 levels), the chunk order is
//     XORed with p mod 8, so the 8 lanes of a row read 8 different bank groups.
//
// One CTA per SM (at most), 768 threads:
//   warp 0       bulk copies: the tile's packed rows, scales and zero points
//   warp 1       allocates 512 TMEM columns; one lane issues the MMAs
//   warps 4-7    epilogue, one per TMEM lane quarter
//   warps 8-23   unpack: four warps per lane quarter take turns over 64-level units
// TMEM: [0, 256) accumulators (256 / N of them), [256, 512) eight A-operand slots of 32
// columns.  Every wait is bounded (common.cuh); after a timeout the CTA drains its
// copies and MMAs, frees TMEM and exits with W4_ERR_TIMEOUT recorded.
#pragma once

#include "gemm_tcgen05.cuh"

namespace w4 {
namespace gemv_tc {

constexpr int NUM_THREADS = 768;
constexpr int EPI_WARP0 = 4;
constexpr int DEQ_WARP0 = 8;
constexpr int DQ = 4;                          // unpack warps per TMEM lane quarter
constexpr int NUM_DEQ_WARPS = 4 * DQ;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_REGION = 256;
constexpr uint32_t SLOT_COLS = 32;             // 64 levels per lane (4 MMA steps)
constexpr int NSLOT = 8;
constexpr int MAX_STAGES = 8;
constexpr int MAX_SETS = 8;
constexpr int MT_MAX = 16;
constexpr int B_MAX_BYTES = 128 * 1024;        // activations resident in shared memory
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr int NUM_BARS = 2 * MAX_STAGES + 2 * NSLOT + 2 * MAX_SETS + 2;

struct Params {
    const __nv_bfloat16 *A;
    const uint8_t *qweight;
    const __half *scales;
    const uint8_t *zeros;
    __nv_bfloat16 *Y;
    int M, N, K;
    int MT;           // activation rows in the B operand (M rounded up)
    int P;            // parts per row (8 or 16)
    int stages;       // shared-memory stages (one tile each)
    int nset;         // accumulators in TMEM
    int tiles;        // ceil(N / R)
    WaitParams wait;
};

__host__ __device__ inline int up128(int x) { return (x + 127) / 128 * 128; }
__host__ __device__ inline int b_bytes(int K, int MT) { return MT * K * 2; }
__host__ __device__ inline int stage_w_bytes(int K, int P) { return up128((128 / P) * (K / 2)); }
__host__ __device__ inline int stage_s_bytes(int K, int P) { return up128((128 / P) * (K / 128) * 2); }
__host__ __device__ inline int stage_bytes(int K, int P) {
    return stage_w_bytes(K, P) + stage_s_bytes(K, P) + up128((128 / P) * (K / 128));
}
__host__ __device__ inline int smem_bytes(int K, int P, int MT, int stages) {
    return b_bytes(K, MT) + stages * stage_bytes(K, P) + NUM_BARS * 8 + 16 + 1024;
}

// One packed word (levels k0..k7, k_j in bits [4j, 4j+4)) -> four bf16 pairs
// ((k_j - zp) * s, (k_{j+4} - zp) * s): exact subtraction, one rounding multiply.
__device__ __forceinline__ void unpack_word(uint32_t x, uint32_t zz2, uint32_t s2, uint32_t *o) {
    const uint32_t magic = 0x43004300u, mask = 0x000F000Fu;  // bf16 (128, 128); ulp 1
    o[0] = gemm::bf16x2_mul(gemm::bf16x2_sub(gemm::lop3_and_or(x, mask, magic), zz2), s2);
    o[1] = gemm::bf16x2_mul(gemm::bf16x2_sub(gemm::lop3_and_or(x >> 4, mask, magic), zz2), s2);
    o[2] = gemm::bf16x2_mul(gemm::bf16x2_sub(gemm::lop3_and_or(x >> 8, mask, magic), zz2), s2);
    o[3] = gemm::bf16x2_mul(gemm::bf16x2_sub(gemm::lop3_and_or(x >> 12, mask, magic), zz2), s2);
}

__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

// v[p] for a lane-dependent p in [0, 16), by a 4-level select tree.
__device__ __forceinline__ float pick16(const uint32_t (&v)[16], int p) {
    uint32_t a[8], b[4], c[2];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (p & 1) ? v[2 * i + 1] : v[2 * i];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = (p & 2) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
    for (int i = 0; i < 2; ++i) c[i] = (p & 4) ? b[2 * i + 1] : b[2 * i];
    return __uint_as_float((p & 8) ? c[1] : c[0]);
}

__device__ __forceinline__ uint32_t bf16_pair_of_half(unsigned short h) {
    const uint32_t b = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(
        __half2float(__ushort_as_half(h)))));
    return b | (b << 16);
}

__global__ void __launch_bounds__(NUM_THREADS, 1) w4a16_skinny_tc_kernel(const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int K = p.K, P = p.P, KP = K / P, UPT = KP / 64, MT = p.MT, NBr = MT * P;
    const int R = 128 / P, ng = K / 128, row_bytes = K / 2;
    const int S = p.stages;
    const int sb = stage_bytes(K, P), swb = stage_w_bytes(K, P), ssb = stage_s_bytes(K, P);
    uint8_t *bsm = smem;                                   // B operand (activations)
    uint8_t *ring = smem + b_bytes(K, MT);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + static_cast<size_t>(S) * sb);
    uint64_t *full = bars;
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *a_full = empty + MAX_STAGES;
    uint64_t *a_empty = a_full + NSLOT;
    uint64_t *acc_full = a_empty + NSLOT;
    uint64_t *acc_empty = acc_full + MAX_SETS;
    uint64_t *mma_done = acc_empty + MAX_SETS;
    uint64_t *never = mma_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long tmo = p.wait.timeout_ns;
    const int t_begin = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.tiles / gridDim.x);
    const int t_end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.tiles / gridDim.x);
    const int nt = t_end - t_begin;

    const uint64_t pol_w = policy_evict_first();
    // Copies of tile lt (packed rows, scales, zero points) into its stage, completing on
    // the stage's full barrier.
    auto issue_tile = [&](int lt) {
        const int stage = lt % S;
        const int r0 = (t_begin + lt) * R;
        const int rows = min(R, p.N - r0);
        uint8_t *st = ring + static_cast<size_t>(stage) * sb;
        const uint32_t wbytes = static_cast<uint32_t>(rows) * row_bytes;
        const uint32_t sbytes = static_cast<uint32_t>(rows) * ng * 2;
        const uint32_t zbytes = static_cast<uint32_t>(rows) * ng;
        mbar_arrive_expect_tx(&full[stage], wbytes + sbytes + zbytes);
        bulk_copy_g2s(st, p.qweight + static_cast<int64_t>(r0) * row_bytes, wbytes, &full[stage], pol_w);
        bulk_copy_g2s(st + swb, p.scales + static_cast<int64_t>(r0) * ng, sbytes, &full[stage], pol_w);
        bulk_copy_g2s(st + swb + ssb, p.zeros + static_cast<int64_t>(r0) * ng, zbytes, &full[stage], pol_w);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NUM_DEQ_WARPS);
        }
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&a_full[s], 4);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < p.nset; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 4);
        }
        mbar_init(mma_done, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
        // The first stages go out before the activations are laid out: the weights do
        // not depend on them, and their DRAM latency then overlaps that work.
        for (int lt = 0; lt < min(S, nt); ++lt) issue_tile(lt);
    }
    if (warp == 1) {
        gemm::tmem_alloc(tmem_slot, TMEM_COLS);
        gemm::tmem_relinquish();
    }
    // B operand: row n = m * P + p holds row m's activations of part p in MMA K order,
    // as K-major 128-byte-swizzled atoms of NBr rows x 64 levels.  Rows m >= M are zero.
    // Each thread issues all its loads before any store, so the latency is paid once.
    {
        constexpr int BATCH = 8;
        const int total = MT * (K / 8);
        for (int base = 0; base < total; base += NUM_THREADS * BATCH) {
            uint4 nat[BATCH];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int idx = base + b * NUM_THREADS + threadIdx.x;
                const int m = idx / (K / 8);
                nat[b] = make_uint4(0, 0, 0, 0);
                if (idx < total && m < p.M)
                    nat[b] = __ldg(reinterpret_cast<const uint4 *>(p.A) + idx);  // A row-major [M, K]
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int idx = base + b * NUM_THREADS + threadIdx.x;
                if (idx >= total) continue;
                const int m = idx / (K / 8);
                const int k = (idx - m * (K / 8)) * 8;
                const int part = k / KP, kl = k - part * KP;
                const int pk = part & 7;
                const int win = kl >> 8, pc = (kl & 255) >> 5, wi = (kl & 31) >> 3;
                const int c = win * 8 + (pc ^ pk);
                const int s = 2 * c + (wi >> 1);
                const int ch = (s & 3) * 2 + (wi & 1);
                const int n = m * P + part;
                uint4 pr;
                pr.x = gemm::prmt(nat[b].x, nat[b].z, 0x5410u);  // (a0, a4)
                pr.y = gemm::prmt(nat[b].x, nat[b].z, 0x7632u);  // (a1, a5)
                pr.z = gemm::prmt(nat[b].y, nat[b].w, 0x5410u);  // (a2, a6)
                pr.w = gemm::prmt(nat[b].y, nat[b].w, 0x7632u);  // (a3, a7)
                *reinterpret_cast<uint4 *>(bsm + (s >> 2) * (NBr * 128) + n * 128 + ((ch ^ (n & 7)) << 4)) = pr;
            }
        }
    }
    fence_proxy_async_smem();
    gemm::tc_fence_before();
    __syncthreads();
    gemm::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer: packed rows, scales and zero points per tile ----------------
        if (lane == 0) {
            int issued_parity[MAX_STAGES];
#pragma unroll
            for (int s = 0; s < MAX_STAGES; ++s) issued_parity[s] = s < min(S, nt) ? 0 : -1;
            bool ok = true;
            for (int lt = min(S, nt); lt < nt; ++lt) {
                const int stage = lt % S;
                const uint32_t phase = static_cast<uint32_t>(lt / S) & 1u;
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                issue_tile(lt);
#pragma unroll
                for (int s = 0; s < MAX_STAGES; ++s)
                    if (s == stage) issued_parity[s] = static_cast<int>(phase);
            }
            if (!ok) {
#pragma unroll
                for (int s = 0; s < MAX_STAGES; ++s)
                    if (issued_parity[s] >= 0)
                        gemm::mbar_wait_drain(&full[s], static_cast<uint32_t>(issued_parity[s]), tmo);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = gemm::make_idesc(static_cast<uint32_t>(NBr));
            const uint32_t b_base = smem_addr(bsm);
            const uint32_t atom = static_cast<uint32_t>(NBr * 128);
            bool ok = true;
            if (p.wait.stall) ok = mbar_wait(never, 0, abort_flag, tmo);  // test hook
            for (int lt = 0; ok && lt < nt; ++lt) {
                const int set = lt % p.nset;
                const uint32_t sphase = static_cast<uint32_t>(lt / p.nset) & 1u;
                if (!mbar_wait(&acc_empty[set], sphase ^ 1u, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                gemm::tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(set * NBr);
                for (int v = 0; v < UPT; ++v) {
                    const int u = lt * UPT + v;
                    const int slot = u % NSLOT;
                    if (!mbar_wait(&a_full[slot], static_cast<uint32_t>(u / NSLOT) & 1u, abort_flag, tmo)) {
                        ok = false;
                        break;
                    }
                    gemm::tc_fence_after();
                    const uint32_t a_tmem = tmem_base + ACC_REGION + static_cast<uint32_t>(slot) * SLOT_COLS;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int s = 4 * v + i;
                        gemm::umma_tmem_a(d_tmem, a_tmem + 8 * i,
                                          gemm::sw128_desc(b_base + static_cast<uint32_t>(s >> 2) * atom + (s & 3) * 32),
                                          idesc, s != 0 ? 1u : 0u);
                    }
                    gemm::umma_commit(&a_empty[slot]);
                }
                if (!ok) break;
                gemm::umma_commit(&acc_full[set]);
            }
            gemm::umma_commit(mma_done);
            gemm::mbar_wait_drain(mma_done, 0, tmo);
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + 4) {
        // ---------------- epilogue: per activation row, own part's column, part sums ----------------
        const int quarter = warp & 3;
        const int li = quarter * 32 + lane;
        const int r = li / P, part = li % P;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        for (int lt = 0; lt < nt; ++lt) {
            const int set = lt % p.nset;
            const uint32_t sphase = static_cast<uint32_t>(lt / p.nset) & 1u;
            const int row = (t_begin + lt) * R + r;
            const bool valid = row < p.N;
            if (!gemm::warp_wait(&acc_full[set], sphase, abort_flag, tmo)) break;
            gemm::tc_fence_after();
            float y[MT_MAX];
#pragma unroll
            for (int m = 0; m < MT_MAX; ++m) {
                y[m] = 0.0f;
                if (m < p.M) {
                    uint32_t v[16];
                    // columns m * P .. m * P + 15 (the upper half unused when P = 8)
                    tmem_ld_16cols(tmem_base + lane_addr + static_cast<uint32_t>(set * NBr + m * P), v);
                    gemm::tmem_wait_ld();
                    y[m] = pick16(v, part);
                }
            }
            gemm::tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[set]);
#pragma unroll
            for (int m = 0; m < MT_MAX; ++m) {
                if (m < p.M) {
                    float s = y[m];
                    for (int o = P >> 1; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    if (part == 0 && valid) p.Y[static_cast<int64_t>(m) * p.N + row] = __float2bfloat16_rn(s);
                }
            }
        }
    } else if (warp >= DEQ_WARP0) {
        // ---------------- unpack packed W -> TMEM A slots ----------------
        const int quarter = warp & 3;
        const int d = (warp - DEQ_WARP0) >> 2;
        const int li = quarter * 32 + lane;
        const int r = li / P, part = li % P, pk = part & 7;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int part_off = r * row_bytes + part * (KP / 2);
        const int Gp = KP / 128;
        bool ok = true;
        for (int lt = 0; ok && lt < nt; ++lt) {
            const int stage = lt % S;
            const uint32_t phase = static_cast<uint32_t>(lt / S) & 1u;
            const uint8_t *st = ring + static_cast<size_t>(stage) * sb;
            const unsigned short *ss = reinterpret_cast<const unsigned short *>(st + swb);
            const uint8_t *zz = st + swb + ssb;
            // Units v of this tile with (lt * UPT + v) % DQ == d (at least one, UPT >= 4).
            const int v0 = ((d - (lt * UPT) % DQ) + DQ) % DQ;
            if (!gemm::warp_wait(&full[stage], phase, abort_flag, tmo)) break;
            for (int v = v0; v < UPT; v += DQ) {
                const int u = lt * UPT + v;
                const int slot = u % NSLOT;
                if (!gemm::warp_wait(&a_empty[slot], (static_cast<uint32_t>(u / NSLOT) & 1u) ^ 1u, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                gemm::tc_fence_after();
                const int win = v >> 2, cc0 = (v & 3) * 2;
                const uint8_t *wbase = st + part_off + win * 128;
                const uint4 x0 = *reinterpret_cast<const uint4 *>(wbase + ((cc0 ^ pk) << 4));
                const uint4 x1 = *reinterpret_cast<const uint4 *>(wbase + (((cc0 + 1) ^ pk) << 4));
                // The two chunks lie in one 128-group of the row.
                const int g = part * Gp + 2 * win + ((cc0 >> 2) ^ (pk >> 2));
                const uint32_t zb = 0x4300u + static_cast<uint32_t>(zz[r * ng + g]);  // bf16(128 + zp), zp < 128
                const uint32_t zz2 = zb | (zb << 16);
                const uint32_t s2 = bf16_pair_of_half(ss[r * ng + g]);
                uint32_t o[32];
                unpack_word(x0.x, zz2, s2, o + 0);
                unpack_word(x0.y, zz2, s2, o + 4);
                unpack_word(x0.z, zz2, s2, o + 8);
                unpack_word(x0.w, zz2, s2, o + 12);
                unpack_word(x1.x, zz2, s2, o + 16);
                unpack_word(x1.y, zz2, s2, o + 20);
                unpack_word(x1.z, zz2, s2, o + 24);
                unpack_word(x1.w, zz2, s2, o + 28);
                tmem_st_32cols(tmem_base + lane_addr + ACC_REGION + static_cast<uint32_t>(slot) * SLOT_COLS, o);
                gemm::tmem_wait_st();
                gemm::tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[slot]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
        }
    }

    gemm::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        gemm::tc_fence_after();
        gemm::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Parts per row: 16 when K is a multiple of 4096 and M <= 8, else 8 when K is a
// multiple of 2048 (keeping N = MT * P <= 128, so two accumulators fit), or 0.
__host__ inline int parts_for(int64_t K, int64_t M) {
    if (K % 4096 == 0 && M <= 8) return 16;
    if (K % 2048 == 0) return 8;
    return 0;
}

}  // namespace gemv_tc
}  // namespace w4
