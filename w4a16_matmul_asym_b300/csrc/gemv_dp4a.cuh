// gemv_dp4a.cuh -- W4A16 decode GEMV (M = 1) on integer dot products.
//
// Computes y[n] = sum_k a[k] * (q[n,k] - zp[n,k/128]) * s16[n,k/128]: the fused
// dequantize-matmul of "Build a GPTQ INT4 Quantization Engine in Python/NumPy"
// (Step 5) with the dequantization of "From Scratch: Building a GPTQ INT4 Quantizer in
// Pure Python" (Step 4), for one activation row.
//
// Why integers: at HBM speed an SM must consume about 50 packed levels per clock, and
// every CUDA-core instruction slot counts.  With the activations turned once into
// integer digits, 8 levels cost 3 unpacking instructions and 6 dp4a, against 7 + 8 for
// the bf16 multiply-add form; the tensor cores do not help here (one MMA instruction
// per 128 x 16 weights, whatever N is, is far too few weights per clock).
//
// Activations as exact integers.  A bf16 value is sig * 2^(E - 134) with an 8-bit
// significand sig (exponent field E, E = 1 for subnormals).  Per 128-group let Emax be
// the largest E of its nonzero finite elements; every element with E >= Emax - 12 is
// exactly v * 2^(Emax - 146) with v = +-sig << (E - Emax + 12), |v| < 2^20.  v is kept
// as three byte digits v = d2 2^16 + d1 2^8 + d0 (d0, d1 unsigned, d2 signed), grouped
// per packed word into the even and odd levels, and dp4a gives exact integer sums
//   t = sum_k v_k q_k - zp sum_k v_k        (|t| < 2^31)
// so a lane's partial is (float(t) * s16) * 2^(Emax - 146).  Elements further below
// the group maximum, and infinities / NaNs, are left out of v (v = 0) and kept in a
// residual array; the lane that owns one adds s16 * (a_k * (q_k - zp)) in fp32, its
// level byte loaded at the start of the stage so the latency hides under the dot
// products (typical activations have none or a handful).  Every product is therefore exact: the
// only roundings are float(t), fp32 multiplies and fp32 sums.
//
// One CTA per SM owns a contiguous band of rows:
//   warps 0..7   consumers.  Lane = one 128-group (or half of one when K = 2048)
//                of the row, its digits in registers; WR = ceil(groups / 32) warps
//                share a row.  Each warp takes RB = 2 rows per stage, releases the
//                stage as soon as it has read it, and writes one fp32 partial per lane
//                and row to a small ring of reduction slots.
//   warp 8       producer: first the activations (one bulk copy, ahead of every
//                weight byte), then each stage's packed rows, scales and zero points,
//                three 1-D bulk copies (the rows of a band are contiguous in all three).
//   warp 9       epilogue: per slot and row, the sum of the partials (fixed order),
//                bf16 rounding and a coalesced store of y.
// Every wait is bounded (common.cuh); after a timeout the CTA drains its copies and
// exits with W4_ERR_TIMEOUT recorded.
//
// W4A8 ("Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization with
// Per-Channel Scale", Step 5): with int8 activations (I8) the digits are the activations
// themselves, one signed byte per level, so the conversion reduces to a byte permute,
// there are no residuals, two dp4a cover 8 levels, and the epilogue multiplies the
// row's sum by the token's activation scale before rounding.
#pragma once

#include "common.cuh"
#include "prefetch.cuh"

namespace w4 {
namespace gemv_dp4a {

constexpr int CW = 8;                      // consumer warps
constexpr int RB = 2;                      // rows per consumer warp per stage
constexpr int PROD_WARP = CW;
constexpr int EPI_WARP = CW + 1;
constexpr int NUM_THREADS = (CW + 2) * 32;
constexpr int MAX_STAGES = 12;
constexpr int RS = 4;                      // reduction slots
constexpr int SMEM_LIMIT = 227 * 1024;

struct Params {
    const void *A;     // bf16 [K], or int8 [K] (I8)
    const float *row_scale;  // I8: the activation scale a_scale[0]
    const uint8_t *qweight;
    const __half *scales;
    const uint8_t *zeros;
    __nv_bfloat16 *Y;
    int N, K;
    int WR;            // warps per row
    int rows_per_cta;  // band size (the last CTA may get fewer)
    int stages;
    WaitParams wait;
};

__host__ __device__ inline int up128(int x) { return (x + 127) / 128 * 128; }

// Shared-memory layout, all offsets 128-byte aligned.
template <int H>
struct Layout {
    static constexpr int WP = 16 / H;              // packed words per lane
    static constexpr int PAD = (H == 1) ? 100 : 52;  // digit words per lane slot (96 / 48 used)
    int K, ng, R, S, WR;
    int stage_w, stage_s, stage_b;                 // W, scales, whole stage
    int off_ring, off_red, off_dig, off_sv, off_csc, off_res, off_cmask, off_bar, total;
    __host__ __device__ Layout(int K_, int WR_, int S_) : K(K_), ng(K_ / 128), R((CW / WR_) * RB), S(S_), WR(WR_) {
        stage_w = up128(R * (K / 2));
        stage_s = up128(R * ng * 2);
        stage_b = stage_w + stage_s + up128(R * ng);
        const int pieces = 32 * WR;                // lane slots (>= ng * H)
        off_ring = 0;
        off_red = off_ring + S * stage_b;
        off_dig = off_red + up128(RS * R * (32 * WR + 1) * 4);
        off_sv = off_dig + up128(pieces * PAD * 4);
        off_csc = off_sv + up128((K / 16) * 4);   // one digit sum per 16-level segment
        off_res = off_csc + up128(ng * 4);         // activations, then their residuals
        off_cmask = off_res + up128(K * 2);
        off_bar = off_cmask + up128((K / 32) * 4);
        total = off_bar + (2 * MAX_STAGES + 2 * RS + 2) * 8 + 16;
    }
    // Fixed part (everything but the ring), for sizing the ring.
    __host__ __device__ int fixed() const { return total - S * stage_b; }
};

// Lane 0 waits (bounded), the result is broadcast, the warp leaves converged.  (The
// vote-based warp_mbar_wait of common.cuh measured slower here: this kernel's epilogue
// warp waits microseconds at a time, and 32 polling lanes compete with the consumers'
// shared-memory traffic.)
__device__ __forceinline__ bool warp_wait_full_bounded(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                       unsigned long long tmo) {
    int ok = 1;
    if (lane_id() == 0) ok = mbar_wait(bar, parity, abort_flag, tmo) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Lane-wise maximum of two pairs of unsigned 16-bit values.
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// 2^e as fp32 for e in [-149, 127] (subnormal below -126), built from bits.
__device__ __forceinline__ float pow2f(int e) {
    if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    return __uint_as_float(1u << (e + 149));
}

// Chunk (32 levels) read by lane l at step j: rotated so that the 8 lanes of a quarter
// warp read 8 different 16-byte bank groups.
template <int H>
__device__ __forceinline__ int lane_rot(int l) {
    return H == 1 ? ((l >> 1) & 3) : ((l >> 2) & 1);
}

template <int H, bool I8>
__global__ void __launch_bounds__(NUM_THREADS, 1) w4a16_gemv_dp4a_kernel(const Params p) {
    constexpr int WP = Layout<H>::WP;
    constexpr int NCH = WP / 4;                    // 32-level chunks per lane
    constexpr int PAD = Layout<H>::PAD;
    extern __shared__ __align__(128) uint8_t smem[];
    const Layout<H> L(p.K, p.WR, p.stages);
    const int K = p.K, ng = K >> 7, row_bytes = K >> 1, R = L.R, S = L.S, WR = p.WR;
    const int red_stride = 32 * WR + 1;
    uint8_t *ring = smem + L.off_ring;
    float *red = reinterpret_cast<float *>(smem + L.off_red);
    uint32_t *dig = reinterpret_cast<uint32_t *>(smem + L.off_dig);
    int *svs = reinterpret_cast<int *>(smem + L.off_sv);          // [K / 16] digit sums
    // Per-segment exponent maxima, only during the conversion: they share the reduction
    // ring (RS * R * (32 WR + 1) floats >= 8 KB >= K / 16 words), untouched until then.
    uint32_t *lmx = reinterpret_cast<uint32_t *>(smem + L.off_red);
    unsigned short *cmask16 = reinterpret_cast<unsigned short *>(smem + L.off_cmask);
    float *cscs = reinterpret_cast<float *>(smem + L.off_csc);
    unsigned short *res = reinterpret_cast<unsigned short *>(smem + L.off_res);
    uint32_t *cmask = reinterpret_cast<uint32_t *>(smem + L.off_cmask);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.off_bar);
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *red_full = empty + MAX_STAGES;
    uint64_t *red_empty = red_full + RS;
    uint64_t *a_bar = red_empty + RS;
    uint64_t *never = a_bar + 1;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(never + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long tmo = p.wait.timeout_ns;
    const int n_begin = blockIdx.x * p.rows_per_cta;
    const int n_end = min(p.N, n_begin + p.rows_per_cta);
    const int num_stages = (max(0, n_end - n_begin) + R - 1) / R;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        for (int s = 0; s < RS; ++s) {
            mbar_init(&red_full[s], CW);
            mbar_init(&red_empty[s], 1);
        }
        mbar_init(a_bar, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // On bands of 96 KB or more, the first 32 KB of weights start towards L2 while the
    // preceding kernel drains (a hint that reads nothing into the CTA, prefetch.cuh).
    // Measured 7.51 -> 7.06 us on 11008 x 4096 and 9.24 -> 8.74 us on 14336 x 4096; on the
    // 57 KB bands of 4096 x 4096 it cost 5 %, hence the floor.
    if (threadIdx.x == 0 && static_cast<int64_t>(n_end - n_begin) * (p.K / 2) >= 98304)
        prefetch_weight_band_l2(p.qweight, p.scales, p.zeros, n_begin, n_end, p.K, 32768);
    pdl_wait_then_release();   // no global memory is read into the CTA before this point

    if (warp == PROD_WARP) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued_parity[MAX_STAGES];
#pragma unroll
            for (int s = 0; s < MAX_STAGES; ++s) issued_parity[s] = -1;
            bool ok = true;
            const uint32_t a_bytes = static_cast<uint32_t>(K) * (I8 ? 1u : 2u);
            mbar_arrive_expect_tx(a_bar, a_bytes);
            bulk_copy_g2s(res, p.A, a_bytes, a_bar, policy_evict_last());
            for (int lt = 0; lt < num_stages; ++lt) {
                const int stage = lt % S;
                const uint32_t phase = static_cast<uint32_t>(lt / S) & 1u;
                if (!mbar_wait_polite(&empty[stage], phase ^ 1u, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                const int r0 = n_begin + lt * R;
                const int rows = min(R, n_end - r0);
                uint8_t *st = ring + static_cast<size_t>(stage) * L.stage_b;
                const uint32_t wb = static_cast<uint32_t>(rows) * row_bytes;
                const uint32_t sb = static_cast<uint32_t>(rows) * ng * 2;
                const uint32_t zb = static_cast<uint32_t>(rows) * ng;
                mbar_arrive_expect_tx(&full[stage], wb + sb + zb);
                bulk_copy_g2s(st, p.qweight + static_cast<int64_t>(r0) * row_bytes, wb, &full[stage], pol);
                bulk_copy_g2s(st + L.stage_w, p.scales + static_cast<int64_t>(r0) * ng, sb, &full[stage], pol);
                bulk_copy_g2s(st + L.stage_w + L.stage_s, p.zeros + static_cast<int64_t>(r0) * ng, zb,
                              &full[stage], pol);
#pragma unroll
                for (int s = 0; s < MAX_STAGES; ++s)
                    if (s == stage) issued_parity[s] = static_cast<int>(phase);
            }
            if (!ok) {
                // Every copy this thread issued lands before the CTA exits.
                const unsigned long long t0 = globaltimer_ns();
                while (!mbar_try_wait(smem_addr(a_bar), 0u))
                    if (globaltimer_ns() - t0 > tmo) break;
#pragma unroll
                for (int s = 0; s < MAX_STAGES; ++s) {
                    if (issued_parity[s] < 0) continue;
                    while (!mbar_try_wait(smem_addr(&full[s]), static_cast<uint32_t>(issued_parity[s])))
                        if (globaltimer_ns() - t0 > tmo) break;
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- activations -> digits (all non-producer warps) ----------------
        // One thread per 16-level segment (two packed words).  No warp shuffles: the
        // group maximum goes through shared memory (each segment's maximum, a barrier,
        // then the eight of its group), and each segment stores its own digit sum and
        // left-out flags, which the consumers combine per lane.
        const int nconv = (CW + 1) * 32;
        const int cw_id = warp < CW ? warp : CW;   // epilogue warp takes the last slot
        const bool have_a = warp_wait_full_bounded(a_bar, 0, abort_flag, tmo);
        for (int sg = cw_id * 32 + lane; I8 && have_a && sg < K / 16; sg += nconv) {
            // int8 activations: the digit words are byte permutes (levels 0 2 4 6 and
            // 1 3 5 7 of each packed word), one signed digit, no residuals.
            const uint4 x = reinterpret_cast<const uint4 *>(res)[sg];
            uint32_t dw[2][6] = {{0, 0, 0, 0, 0, 0}, {0, 0, 0, 0, 0, 0}};
            dw[0][0] = byte_perm(x.x, x.y, 0x6420u);
            dw[0][3] = byte_perm(x.x, x.y, 0x7531u);
            dw[1][0] = byte_perm(x.z, x.w, 0x6420u);
            dw[1][3] = byte_perm(x.z, x.w, 0x7531u);
            int vsum = 0;
            const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) vsum = __dp4a(static_cast<int>(xw[i]), 0x01010101, vsum);
            const int g = sg >> 3;
            const int piece = g * H + (sg & 7) / (8 / H);
            const int wi = ((sg & 7) % (8 / H)) * 2;
            const int cpos = wi >> 2;
            const int slot = (cpos - lane_rot<H>(piece & 31)) & (NCH - 1);
            uint4 *dst = reinterpret_cast<uint4 *>(dig + piece * PAD + (slot * 4 + (wi & 3)) * 6);
            dst[0] = make_uint4(dw[0][0], dw[0][1], dw[0][2], dw[0][3]);
            dst[1] = make_uint4(dw[0][4], dw[0][5], dw[1][0], dw[1][1]);
            dst[2] = make_uint4(dw[1][2], dw[1][3], dw[1][4], dw[1][5]);
            cmask16[sg] = 0;
            svs[sg] = vsum;
            if ((sg & 7) == 0) cscs[g] = 1.0f;
        }
        if constexpr (!I8) {
            // Pass 1: each segment's maximum of the exponent|mantissa bits (infinities
            // and NaNs included: such a group sends all its finite elements to the
            // residual path).
            for (int sg = cw_id * 32 + lane; have_a && sg < K / 16; sg += nconv) {
                const uint4 *src = reinterpret_cast<const uint4 *>(res) + sg * 2;
                const uint4 x0 = src[0], x1 = src[1];
                uint32_t mx = vmax_u16x2(x0.x & 0x7FFF7FFFu, x0.y & 0x7FFF7FFFu);
                mx = vmax_u16x2(mx, x0.z & 0x7FFF7FFFu);
                mx = vmax_u16x2(mx, x0.w & 0x7FFF7FFFu);
                mx = vmax_u16x2(mx, x1.x & 0x7FFF7FFFu);
                mx = vmax_u16x2(mx, x1.y & 0x7FFF7FFFu);
                mx = vmax_u16x2(mx, x1.z & 0x7FFF7FFFu);
                mx = vmax_u16x2(mx, x1.w & 0x7FFF7FFFu);
                lmx[sg] = max(mx & 0xFFFFu, mx >> 16);
            }
            asm volatile("bar.sync 2, %0;" ::"r"((CW + 1) * 32) : "memory");
            // Pass 2: the digits.
            for (int sg = cw_id * 32 + lane; have_a && sg < K / 16; sg += nconv) {
                uint32_t w[8];                     // 16 bf16, two per word, natural order
                {
                    const uint4 *src = reinterpret_cast<const uint4 *>(res) + sg * 2;
                    const uint4 x0 = src[0], x1 = src[1];
                    w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
                    w[4] = x1.x; w[5] = x1.y; w[6] = x1.z; w[7] = x1.w;
                }
                const int g = sg >> 3;             // 8 segments per group
                uint32_t mx;
                {
                    const uint4 m0 = reinterpret_cast<const uint4 *>(lmx)[2 * g];
                    const uint4 m1 = reinterpret_cast<const uint4 *>(lmx)[2 * g + 1];
                    mx = max(max(max(m0.x, m0.y), max(m0.z, m0.w)), max(max(m1.x, m1.y), max(m1.z, m1.w)));
                }
                const int emax = max(static_cast<int>(mx >> 7), 1);  // exponent field, >= 1
                // v = a * 2^c, c = 146 - emax, |v| < 2^20; exact iff |a| >= 2^(emax - 139).
                const int c = 146 - emax;
                const float c1 = pow2f(min(c, 127)), c2 = pow2f(max(c - 127, 0));
                const float thr = pow2f(emax - 139);
                int v[16];
                uint32_t flag = 0;
                int vsum = 0;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a = __uint_as_float((i & 1) ? (w[i >> 1] & 0xFFFF0000u) : (w[i >> 1] << 16));
                    const float tt = __fmaf_rn(__fmul_rn(a, c1), c2, 12582912.0f);  // 1.5 * 2^23: round to integer
                    const int vi = __float_as_int(tt) - 0x4B400000;
                    const float m = fabsf(a);
                    const bool left_out = !(m <= 3.402823466e38f) || (m != 0.0f && m < thr);  // inf / NaN, or too small
                    v[i] = left_out ? 0 : vi;
                    vsum += v[i];
                    flag |= static_cast<uint32_t>(left_out) << i;
                }
                // Digit words of each packed word: even levels (0, 2, 4, 6), odd levels
                // (1, 3, 5, 7); byte j of digit word d is byte d of v of the j-th level.
                uint32_t dw[2][6];
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int par = 0; par < 2; ++par) {
                        const uint32_t va = static_cast<uint32_t>(v[8 * q + par]), vb = static_cast<uint32_t>(v[8 * q + 2 + par]);
                        const uint32_t vc = static_cast<uint32_t>(v[8 * q + 4 + par]), vd = static_cast<uint32_t>(v[8 * q + 6 + par]);
                        const uint32_t lo_ab = byte_perm(va, vb, 0x5140u), lo_cd = byte_perm(vc, vd, 0x5140u);
                        const uint32_t hi_ab = byte_perm(va, vb, 0x0062u), hi_cd = byte_perm(vc, vd, 0x0062u);
                        dw[q][3 * par + 0] = byte_perm(lo_ab, lo_cd, 0x5410u);
                        dw[q][3 * par + 1] = byte_perm(lo_ab, lo_cd, 0x7632u);
                        dw[q][3 * par + 2] = byte_perm(hi_ab, hi_cd, 0x5410u);
                    }
                // Piece (lane slot) of this segment and its place in the lane's rotated order.
                const int piece = g * H + (sg & 7) / (8 / H);
                const int wi = ((sg & 7) % (8 / H)) * 2;  // first packed word within the piece
                const int cpos = wi >> 2;                // chunk within the piece
                const int slot = (cpos - lane_rot<H>(piece & 31)) & (NCH - 1);
                uint4 *dst = reinterpret_cast<uint4 *>(dig + piece * PAD + (slot * 4 + (wi & 3)) * 6);
                dst[0] = make_uint4(dw[0][0], dw[0][1], dw[0][2], dw[0][3]);
                dst[1] = make_uint4(dw[0][4], dw[0][5], dw[1][0], dw[1][1]);
                dst[2] = make_uint4(dw[1][2], dw[1][3], dw[1][4], dw[1][5]);
                // residuals: the bf16 bits of the elements left out of v
                uint32_t rw[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t keep = (((flag >> (2 * i)) & 1u) ? 0x0000FFFFu : 0u) |
                                          (((flag >> (2 * i + 1)) & 1u) ? 0xFFFF0000u : 0u);
                    rw[i] = w[i] & keep;
                }
                uint4 *rdst = reinterpret_cast<uint4 *>(res) + sg * 2;
                rdst[0] = make_uint4(rw[0], rw[1], rw[2], rw[3]);
                rdst[1] = make_uint4(rw[4], rw[5], rw[6], rw[7]);
                cmask16[sg] = static_cast<unsigned short>(flag);
                svs[sg] = vsum;
                if ((sg & 7) == 0) cscs[g] = pow2f(emax - 146);
            }
        }
    }
    if (warp != PROD_WARP) {
        // Named barrier of the non-producer warps: the producer is already streaming.
        asm volatile("bar.sync 1, %0;" ::"r"((CW + 1) * 32) : "memory");
    }

    if (warp < CW) {
        // ---------------- consumers ----------------
        const int rb = warp / WR, wr = warp % WR;
        const int l = lane, piece = wr * 32 + l;
        const bool active = piece < ng * H;
        const int g = piece / H, hh = piece % H;
        const int rot = lane_rot<H>(l);
        uint32_t dg[NCH][4][6];
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(dig + piece * PAD);
#pragma unroll
            for (int i = 0; i < NCH * 6; ++i) {
                const uint4 x = active ? src[i] : make_uint4(0, 0, 0, 0);
                uint32_t *d = &dg[0][0][0] + 4 * i;
                d[0] = x.x;
                d[1] = x.y;
                d[2] = x.z;
                d[3] = x.w;
            }
        }
        // Residual (left-out) elements of this lane's piece, in order: up to four in
        // registers (element index in the piece, value); a lane with more takes a
        // masked slow path for all of them.
        constexpr int PL = 128 / H;                // levels per piece
        const int pbase = g * 128 + hh * PL;       // first level of the piece
        uint32_t lst = 0;
        float af[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        int cnt = 0;
        uint32_t fmc[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            fmc[c] = active ? cmask[(pbase >> 5) + c] : 0u;
            uint32_t m = fmc[c];
            while (m) {
                const int e = c * 32 + __ffs(m) - 1;
                m &= m - 1u;
#pragma unroll
                for (int f = 0; f < 4; ++f)
                    if (cnt == f) {
                        lst |= static_cast<uint32_t>(e) << (8 * f);
                        af[f] = __uint_as_float(static_cast<uint32_t>(res[pbase + e]) << 16);
                    }
                ++cnt;
            }
        }
        if (cnt > 4) {
#pragma unroll
            for (int f = 0; f < 4; ++f) af[f] = 0.0f;
        }
        const int wlist = __reduce_max_sync(0xffffffffu, cnt > 4 ? 0 : cnt);  // warp-uniform
        const bool wslow = __any_sync(0xffffffffu, cnt > 4);
        int sv = 0;                                // sum of v over the lane's piece
        if (active) {
#pragma unroll
            for (int i = 0; i < 8 / H; ++i) sv += svs[piece * (8 / H) + i];
        }
        const float csc = active ? cscs[g] : 0.0f;
        const int wbyte = g * 64 + hh * 32;
        bool ok = true;
        if (p.wait.stall) ok = mbar_wait(never, 0, abort_flag, tmo);  // test hook
        int stage = 0, slot = 0;
        uint32_t phase = 0, sphase = 0;
        for (int lt = 0; ok && lt < num_stages; ++lt) {
            // Every lane polls the barrier itself: no broadcast round trip per stage.
            if (!mbar_wait(&full[stage], phase, abort_flag, tmo)) break;
            const uint8_t *st = ring + static_cast<size_t>(stage) * L.stage_b;
            const unsigned short *ss = reinterpret_cast<const unsigned short *>(st + L.stage_w);
            const uint8_t *zz = st + L.stage_w + L.stage_s;
            // Separate accumulators for even and odd levels: 12 independent dp4a chains.
            uint32_t s0e[RB], s1e[RB], s0o[RB], s1o[RB];
            int s2e[RB], s2o[RB];
            float sf[RB];
            uint32_t zp[RB];
            // Bytes holding the residual elements' levels, loaded now so that their
            // latency hides under the dot products.
            uint32_t qb[4][RB];
#pragma unroll
            for (int f = 0; f < 4; ++f)
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    qb[f][i] = 0;
                    if (f < wlist) {
                        const int e = static_cast<int>((lst >> (8 * f)) & 0xFFu);
                        qb[f][i] = st[(rb * RB + i) * row_bytes + wbyte + (e >> 1)];
                    }
                }
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const int r = rb * RB + i;  // rows past the band hold stale bytes: finite, unused
                s0e[i] = s1e[i] = s0o[i] = s1o[i] = 0;
                s2e[i] = s2o[i] = 0;
                sf[i] = __half2float(__ushort_as_half(ss[r * ng + g]));
                zp[i] = zz[r * ng + g];
            }
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                const int c = (j + rot) & (NCH - 1);
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    const int r = rb * RB + i;
                    const uint4 wv = *reinterpret_cast<const uint4 *>(st + r * row_bytes + wbyte + c * 16);
                    const uint32_t x[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t ev = x[w] & 0x0F0F0F0Fu;
                        const uint32_t od = (x[w] >> 4) & 0x0F0F0F0Fu;
                        if constexpr (I8) {        // one signed digit
                            s2e[i] = dp4a_su(dg[j][w][0], ev, s2e[i]);
                            s2o[i] = dp4a_su(dg[j][w][3], od, s2o[i]);
                        } else {
                            s0e[i] = dp4a_uu(dg[j][w][0], ev, s0e[i]);
                            s1e[i] = dp4a_uu(dg[j][w][1], ev, s1e[i]);
                            s2e[i] = dp4a_su(dg[j][w][2], ev, s2e[i]);
                            s0o[i] = dp4a_uu(dg[j][w][3], od, s0o[i]);
                            s1o[i] = dp4a_uu(dg[j][w][4], od, s1o[i]);
                            s2o[i] = dp4a_su(dg[j][w][5], od, s2o[i]);
                        }
                    }
                }
            }
            // Residual elements: a_k * (q_k - zp), exact, in fp32.
            float rr[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) rr[i] = 0.0f;
#pragma unroll
            for (int f = 0; f < 4; ++f)
                if (f < wlist) {
                    const int sh = static_cast<int>((lst >> (8 * f)) & 1u) * 4;
#pragma unroll
                    for (int i = 0; i < RB; ++i) {
                        const int qv = static_cast<int>((qb[f][i] >> sh) & 15u);
                        rr[i] = __fmaf_rn(af[f], static_cast<float>(qv - static_cast<int>(zp[i])), rr[i]);
                    }
                }
            if (wslow && cnt > 4) {
#pragma unroll 1
                for (int c = 0; c < NCH; ++c) {
                    uint32_t m = c == 0 ? fmc[0] : c == 1 ? fmc[NCH > 1 ? 1 : 0] : c == 2 ? fmc[NCH > 2 ? 2 : 0] : fmc[NCH > 3 ? 3 : 0];
                    while (m) {
                        const int e = c * 32 + __ffs(m) - 1;
                        m &= m - 1u;
                        const float a = __uint_as_float(static_cast<uint32_t>(res[pbase + e]) << 16);
#pragma unroll
                        for (int i = 0; i < RB; ++i) {
                            const int qv = (st[(rb * RB + i) * row_bytes + wbyte + (e >> 1)] >> ((e & 1) * 4)) & 15;
                            rr[i] = __fmaf_rn(a, static_cast<float>(qv - static_cast<int>(zp[i])), rr[i]);
                        }
                    }
                }
            }
            // The stage is consumed: the producer may refill it.
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (!mbar_wait(&red_empty[slot], sphase ^ 1u, abort_flag, tmo)) break;
            float *rd = red + static_cast<size_t>(slot) * R * red_stride;
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const int r = rb * RB + i;
                // sum_k v_k (q_k - zp); intermediate values wrap, the result fits in int32.
                const uint32_t tu = I8 ? static_cast<uint32_t>(s2e[i] + s2o[i]) - zp[i] * static_cast<uint32_t>(sv)
                                       : static_cast<uint32_t>(s2e[i] + s2o[i]) * 65536u + (s1e[i] + s1o[i]) * 256u +
                                             (s0e[i] + s0o[i]) - zp[i] * static_cast<uint32_t>(sv);
                float part = __fmul_rn(__fmul_rn(__int2float_rn(static_cast<int>(tu)), sf[i]), csc);
                part = __fmaf_rn(sf[i], rr[i], part);
                rd[r * red_stride + piece] = active ? part : 0.0f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&red_full[slot]);
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
            if (++slot == RS) {
                slot = 0;
                sphase ^= 1u;
            }
        }
    } else if (warp == EPI_WARP) {
        // ---------------- epilogue ----------------
        const int r = lane;
        int slot = 0;
        uint32_t sphase = 0;
        for (int lt = 0; lt < num_stages; ++lt) {
            const int r0 = n_begin + lt * R;
            const int rows = min(R, n_end - r0);
            int got = 1;
            if (lane == 0) got = mbar_wait(&red_full[slot], sphase, abort_flag, tmo);
            got = __shfl_sync(0xffffffffu, got, 0);
            __syncwarp();
            if (!got) break;
            const float *rd = red + static_cast<size_t>(slot) * R * red_stride;
            if (r < rows) {
                float y = 0.0f;
                for (int j = 0; j < 32 * WR; ++j) y += rd[r * red_stride + j];
                if constexpr (I8) y = __fmul_rn(y, p.row_scale[0]);
                p.Y[r0 + r] = __float2bfloat16_rn(y);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&red_empty[slot]);
            if (++slot == RS) {
                slot = 0;
                sphase ^= 1u;
            }
        }
    }
    __syncthreads();
}

}  // namespace gemv_dp4a
}  // namespace w4
