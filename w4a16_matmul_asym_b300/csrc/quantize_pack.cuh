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
// Symmetric variant ("Build a GPTQ INT4 Quantization Engine in Python/NumPy", Step 2):
//   s  = (absmax == 0) ? 1 : absmax / 7, absmax = max(|min|, |max|)   IEEE division
//   zp = 8, so q = clip(rhe(w / s) + 8, 0, 15) = clip(rhe(w / s), -8, 7) + 8
// and everything after the group parameters is shared.
//
// Layout: the flat group index G = n * (K/128) + g addresses every output directly:
// qweight bytes [64 G, 64 G + 64), scales[G], zeros[G], and W elements
// [128 G, 128 G + 128).  The kernel walks groups as one flat array.
//
// Mapping: LPG lanes own a group (2 for fp16, 4 for fp32), each lane one 128-byte line
// of W (64 fp16 or 32 fp32 elements).  One CTA per SM: a producer warp streams W
// through a 3-stage shared-memory ring with 2-D tensor copies (64 KB per stage: one
// 4 KB block per consumer warp), 128-byte swizzled so that the 8 lanes of a quarter
// warp read 8 different bank groups; the 16 consumer warps copy their lines into
// registers, release the stage at once and quantize from registers.  Up to 192 KB of
// W is in flight per SM.  Min/max: a local tree (on packed halves for fp16) and a 1- or
// 2-step xor-shuffle.  Each lane writes its packed nibbles as 16- or 32-byte
// vector stores; a warp stores 1 KB (fp16) or 512 B (fp32) of qweight contiguously.
//
// The quotient w/s without a divide per element: t = w * fl(1/s) lies within 3 ulp
// of the IEEE quotient x = fl(w/s) (two roundings of 2^-24 relative each, plus x's
// own), i.e. within 1.2e-5 for |x| <= 64.  Only x + zp in [-0.5, 15.5] (|x| < 16)
// escapes the clip, so that bound is the one that matters.
//   level:    lv = sat((t + zp) / 15) with one fma.sat, which also performs the clip
//             to [0, 15]; |15 lv - (t + zp)| < 3e-6 below saturation (the roundings
//             of fl(1/15), of zp fl(1/15) and of the fma, 2^-24 relative each, on
//             values up to 15.5).  With M = 1.5 * 2^23, q = fl(15 lv + M) = M + rhe(15 lv).
//   tie test: e = fl(15 lv - (q - M)) is 15 lv minus its rounding, to 2^-25.  When
//             |e| <= 0.5 - 2^-15, 15 lv is at least 2^-15 = 3.05e-5 from every
//             half-integer, so x + zp (within 1.2e-5 + 3e-6 of 15 lv) rounds to the
//             same integer and q is the exact level.  Words with an element outside
//             that (about 6e-5 of the elements) redo the word with the IEEE division
//             __fdiv_rn.  A saturated lv gives e = 0: the clipped level needs no
//             tie-breaking.
//   packing:  four levels per fp32 lane of an f32x2 pair, 2^23 + q0 + 16 q1 + 256 q2
//             + 4096 q3 (exact), the two 16-bit sums merged with one prmt.
#pragma once

#include "common.cuh"
#include "prefetch.cuh"

namespace w4 {

constexpr float kRoundMagic = 12582912.0f;              // 1.5 * 2^23
constexpr float kTieEdge = 0.499969482421875f;         // 0.5 - 2^-15

// ---- f32x2 helpers (Blackwell packed fp32) ------------------------------------------
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
    float d;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// Exact fp16 -> fp32 widening on the FMA pipe: f32(h) + (-0).
__device__ __forceinline__ float widen_lo(uint32_t h2) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.f16 %0, lo, 0f80000000;\n\t}"
        : "=f"(r) : "r"(h2));
    return r;
}
__device__ __forceinline__ float widen_hi(uint32_t h2) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.f16 %0, hi, 0f80000000;\n\t}"
        : "=f"(r) : "r"(h2));
    return r;
}

struct GroupParams {
    float s;        // fp32 scale
    uint64_t rcp2;  // (fl(1/s), fl(1/s))
    uint64_t mz2;   // (M + zp, M + zp), exact
    float r15;      // fl(1/15)
    float c15;      // fl(zp * fl(1/15))
    float zp;       // zero point (0..15) as float
    bool exact;     // fl(1/s) overflowed (s < ~2^-128): every level by IEEE division
};

template <bool kSym>
__device__ __forceinline__ GroupParams group_params(float mn, float mx) {
    GroupParams p;
    if constexpr (kSym) {
        const float amax = fmaxf(fabsf(mn), fabsf(mx));   // exact
        p.s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 7.0f);
        p.zp = 8.0f;
    } else {
        p.s = (mx == mn) ? 1.0f : __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
        const float x = __fdiv_rn(-mn, p.s);
        // rhe(x) for |x| < 2^22 via the magic add; larger |x| clips anyway.
        const float zq = (fabsf(x) < 4194304.0f) ? __fsub_rn(__fadd_rn(x, kRoundMagic), kRoundMagic) : x;
        p.zp = fminf(fmaxf(zq, 0.0f), 15.0f);
    }
    const float rcp = __frcp_rn(p.s);
    // A scale below about 2^-128 (an fp32 group range under ~4.4e-38, or an absmax
    // under ~2e-38 in the symmetric variant) has no finite reciprocal: t = w * rcp
    // would be +-inf or NaN and the tie test below would not see it.  Such groups
    // take the exact per-element division.
    p.exact = (__float_as_uint(rcp) & 0x7f800000u) == 0x7f800000u;
    const float mz = __fadd_rn(kRoundMagic, p.zp);
    p.rcp2 = f2pack(rcp, rcp);
    p.mz2 = f2pack(mz, mz);
    p.r15 = 0.0666666701436042785644531f;  // fl(1/15)
    p.c15 = __fmul_rn(p.zp, p.r15);
    return p;
}

// Exact reference for one element: kRoundMagic + clip(rhe(w / s) + zp, 0, 15).
__device__ __forceinline__ float level_exact(float w, const GroupParams &p) {
    const float x = __fdiv_rn(w, p.s);
    float v;
    if (fabsf(x) < 4194304.0f) {
        const float k = __fsub_rn(__fadd_rn(x, kRoundMagic), kRoundMagic);  // rhe(x)
        v = __fadd_rn(kRoundMagic, __fadd_rn(k, p.zp));
    } else {
        v = (x > 0.0f) ? kRoundMagic + 15.0f : kRoundMagic;
    }
    return fminf(fmaxf(v, kRoundMagic), kRoundMagic + 15.0f);
}

// Four f32x2 pairs q[j] = M + level (elements j and j + 4) -> one 32-bit word of
// nibbles (element i in bits [4i, 4i+4)): one f32x2 packing chain builds the low and
// the high 16 bits at once; element 0's pair takes M - 2^23 off so the chain carries 2^23.
__device__ __forceinline__ uint32_t pack8(const uint64_t (&q)[4]) {
    const uint64_t M2 = f2pack(kRoundMagic, kRoundMagic);
    const uint64_t M22 = f2pack(4194304.0f, 4194304.0f);  // 2^22: L - 2^22 = 2^23 + q
    uint64_t acc = f2sub(q[0], M22);
    acc = f2fma(f2sub(q[1], M2), f2pack(16.0f, 16.0f), acc);
    acc = f2fma(f2sub(q[2], M2), f2pack(256.0f, 256.0f), acc);
    acc = f2fma(f2sub(q[3], M2), f2pack(4096.0f, 4096.0f), acc);
    float lo, hi;
    f2unpack(acc, lo, hi);
    uint32_t word;
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(word) : "r"(__float_as_uint(lo)), "r"(__float_as_uint(hi)));
    return word;
}

// 8 consecutive elements w[0..7] -> their word by the reciprocal path.  `tie` is set
// when an element falls in the tie window (or the group has no finite reciprocal):
// the word must then be redone by quantize8_exact.
__device__ __forceinline__ uint32_t quantize8_fast(const float (&w)[8], const GroupParams &p, bool &tie) {
    const uint64_t M2 = f2pack(kRoundMagic, kRoundMagic);
    const uint64_t c15x2 = f2pack(15.0f, 15.0f);
    uint64_t q[4];
    tie = p.exact;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t t = f2mul(f2pack(w[j], w[j + 4]), p.rcp2);
        float tlo, thi;
        f2unpack(t, tlo, thi);
        const uint64_t lv = f2pack(fma_sat(tlo, p.r15, p.c15), fma_sat(thi, p.r15, p.c15));
        q[j] = f2fma(lv, c15x2, M2);                             // M + level
        const uint64_t e = f2fma(lv, c15x2, f2sub(M2, q[j]));    // 15 lv - level
        float elo, ehi;
        f2unpack(e, elo, ehi);
        tie |= (fabsf(elo) > kTieEdge) | (fabsf(ehi) > kTieEdge);
    }
    return pack8(q);
}

// The same word with every quotient by IEEE division.
__device__ __forceinline__ uint32_t quantize8_exact(const float (&w)[8], const GroupParams &p) {
    uint64_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = f2pack(level_exact(w[j], p), level_exact(w[j + 4], p));
    return pack8(q);
}

template <bool kF32>
struct QuantCfg {
    static constexpr int kLanesPerGroup = kF32 ? 4 : 2;
    static constexpr int kElemsPerLane = 128 / kLanesPerGroup;   // 32 or 64
    static constexpr int kGroupsPerWarp = 32 / kLanesPerGroup;   // 8 or 16
    static constexpr int kLoads = 8;                             // 16-byte loads per lane
    static constexpr int kWords = kElemsPerLane / 8;             // output words per lane
};

// Elements 8c .. 8c+7 of a lane's 128 bytes of W, widened exactly to fp32.
template <bool kF32>
__device__ __forceinline__ void lane_elems(const uint4 (&cur)[QuantCfg<kF32>::kLoads], int c, float (&w)[8]) {
    if constexpr (kF32) {
        const float *f = reinterpret_cast<const float *>(cur) + 8 * c;
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = f[i];
    } else {
        const uint32_t *u = reinterpret_cast<const uint32_t *>(cur) + 4 * c;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w[2 * i] = widen_lo(u[i]);
            w[2 * i + 1] = widen_hi(u[i]);
        }
    }
}

// One lane's 128 bytes of W (cur, natural order) -> its qweight words; the group's
// scale and zero point are written by the lane with part 0.  g = flat group index.
template <bool kF32, bool kSym>
__device__ __forceinline__ void quantize_lane(const uint4 (&cur)[QuantCfg<kF32>::kLoads], int64_t g,
                                              int part, int64_t total_groups, uint32_t *__restrict__ qw,
                                              __half *__restrict__ scales, uint8_t *__restrict__ zeros) {
    using C = QuantCfg<kF32>;
    // ---- min / max over the group ----
    float mn, mx;
    if constexpr (kF32) {
        const float *f = reinterpret_cast<const float *>(cur);
        mn = f[0];
        mx = f[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) {
            mn = fminf(mn, f[i]);
            mx = fmaxf(mx, f[i]);
        }
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    } else {
        const __half2 *h = reinterpret_cast<const __half2 *>(cur);
        __half2 lo2 = __hmin2(h[0], h[1]), hi2 = __hmax2(h[0], h[1]);
#pragma unroll
        for (int i = 2; i < 32; i += 2) {
            lo2 = __hmin2(lo2, __hmin2(h[i], h[i + 1]));
            hi2 = __hmax2(hi2, __hmax2(h[i], h[i + 1]));
        }
        // (min, -max) in one half2 so one shuffle + one hmin2 combines both.
        const __half mnh = __hmin(__low2half(lo2), __high2half(lo2));
        const __half mxh = __hmax(__low2half(hi2), __high2half(hi2));
        __half2 pk = __halves2half2(mnh, __hneg(mxh));
        const uint32_t pku = *reinterpret_cast<const uint32_t *>(&pk);
        const uint32_t oth = __shfl_xor_sync(0xffffffffu, pku, 1);
        pk = __hmin2(pk, *reinterpret_cast<const __half2 *>(&oth));
        const uint32_t pkb = *reinterpret_cast<const uint32_t *>(&pk);
        mn = widen_lo(pkb);
        mx = -widen_hi(pkb);
    }
    const GroupParams p = group_params<kSym>(mn, mx);

    // ---- quantize and pack, 8 elements per output word ----
    // (Redoing the rare tie-window words in a second loop instead of at once spilled
    // at the 96-register cap of 17 warps and ran 20 % slower.)
    uint32_t words[C::kWords];
#pragma unroll
    for (int c = 0; c < C::kWords; ++c) {
        float w[8];
        lane_elems<kF32>(cur, c, w);
        bool tie;
        words[c] = quantize8_fast(w, p, tie);
        if (tie) words[c] = quantize8_exact(w, p);
    }
    if (g < total_groups) {
        uint4 *dst = reinterpret_cast<uint4 *>(qw + g * 16 + part * C::kWords);
#pragma unroll
        for (int c = 0; c < C::kWords; c += 4)
            dst[c / 4] = make_uint4(words[c], words[c + 1], words[c + 2], words[c + 3]);
        if (part == 0) {
            scales[g] = __float2half_rn(p.s);
            zeros[g] = static_cast<uint8_t>(p.zp);
        }
    }
}

namespace quant {
constexpr int CW = 16;                       // consumer warps
constexpr int NUM_THREADS = (CW + 1) * 32;
constexpr int STAGES = 3;
constexpr int LINES = CW * 32;               // 128-byte lines per stage (one per consumer lane)
constexpr int STAGE_BYTES = LINES * 128;     // 64 KB
constexpr int BOX_LINES = 256;               // tensor-copy box: 128 B x 256 lines
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + (2 * STAGES + 1) * 8 + 1024;
}  // namespace quant

// W viewed as bytes in 128-byte lines: tmW is a 2-D map {128 B, total_lines} with
// 128-byte swizzle.  Stage unit u covers lines [u * LINES, (u + 1) * LINES), i.e.
// groups [u * CW * kGroupsPerWarp, ...); CTA b takes units b, b + gridDim.x, ...
template <bool kF32, bool kSym>
__global__ void __launch_bounds__(quant::NUM_THREADS, 1)
    quantize_pack_kernel(const __grid_constant__ CUtensorMap tmW, int64_t total_groups,
                         uint32_t *__restrict__ qw, __half *__restrict__ scales,
                         uint8_t *__restrict__ zeros, WaitParams wait, const uint8_t *w_bytes) {
    using C = QuantCfg<kF32>;
    using namespace quant;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *never = empty + STAGES;
    __shared__ int abort_flag_s;
    volatile int *abort_flag = &abort_flag_s;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long tmo = wait.timeout_ns;
    constexpr int kLinesPerGroup = C::kLanesPerGroup;
    const int64_t total_lines = total_groups * kLinesPerGroup;
    const int64_t units = (total_lines + LINES - 1) / LINES;
    const int64_t my_units = units > blockIdx.x ? (units - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmW);
    }
    __syncthreads();
    // The CTA's first stage unit (64 KB of W, as bytes) starts towards L2 while the
    // preceding kernel drains: a hint that reads nothing into the CTA (prefetch.cuh).
    // Measured (fp16 W) 13.9 -> 12.6 us on 4096 x 4096, 26.7 -> 25.3 us on 11008 x 4096
    // and 108.4 -> 106.0 us on 28672 x 8192; a second unit added nothing.  The symmetric
    // variant leaves it out: with the prefetch compiled in, its main loop ran 4 % slower
    // on 28672 x 8192 (117.2 against 112.9 us) even when the prefetch was skipped at run
    // time (the code generated for the loop changed), which outweighs its gain on small
    // shapes (14.0 -> 12.8 us on 4096 x 4096).
    if constexpr (!kSym) {
        if (threadIdx.x == CW * 32 && my_units > 0) {
            const int64_t b0 = static_cast<int64_t>(blockIdx.x) * STAGE_BYTES;
            prefetch_l2_range(w_bytes, b0, min(b0 + STAGE_BYTES, total_lines * 128));
        }
    }
    pdl_wait_then_release();   // no global memory is read into the CTA before this point

    if (warp == CW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued_parity[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
            bool ok = true;
            for (int64_t lt = 0; lt < my_units; ++lt) {
                const int stage = static_cast<int>(lt % STAGES);
                const uint32_t phase = static_cast<uint32_t>(lt / STAGES) & 1u;
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, tmo)) {
                    ok = false;
                    break;
                }
                const int64_t line0 = (blockIdx.x + lt * gridDim.x) * LINES;
                // Boxes that start inside the tensor; a box reaching past its end is
                // filled with zeros (and counts in full).
                const int nbox = static_cast<int>(min(static_cast<int64_t>(LINES / BOX_LINES),
                                                      (total_lines - line0 + BOX_LINES - 1) / BOX_LINES));
                uint8_t *st = smem + stage * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(nbox) * BOX_LINES * 128);
                for (int b = 0; b < nbox; ++b)
                    tma_load_2d(st + b * BOX_LINES * 128, &tmW, &full[stage], 0,
                                static_cast<int>(line0 + b * BOX_LINES), pol);
#pragma unroll
                for (int s = 0; s < STAGES; ++s)
                    if (s == stage) issued_parity[s] = static_cast<int>(phase);
            }
            if (!ok) {
                const unsigned long long t0 = globaltimer_ns();
#pragma unroll
                for (int s = 0; s < STAGES; ++s) {
                    if (issued_parity[s] < 0) continue;
                    while (!mbar_try_wait(smem_addr(&full[s]), static_cast<uint32_t>(issued_parity[s])))
                        if (globaltimer_ns() - t0 > tmo) break;
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- consumers ----------------
        const int gsub = lane / C::kLanesPerGroup;  // group within the warp's block
        const int part = lane % C::kLanesPerGroup;  // line within the group
        const int ln = warp * 32 + lane;             // my line within the stage
        bool ok = true;
        if (wait.stall) ok = mbar_wait(never, 0, abort_flag, tmo);  // test hook: nothing signals it
        for (int64_t lt = 0; ok && lt < my_units; ++lt) {
            const int stage = static_cast<int>(lt % STAGES);
            const uint32_t phase = static_cast<uint32_t>(lt / STAGES) & 1u;
            if (!mbar_wait(&full[stage], phase, abort_flag, tmo)) break;
            // Logical 16-byte chunk i of line ln sits at chunk i ^ (ln & 7).
            const uint8_t *line = smem + stage * STAGE_BYTES + ln * 128;
            uint4 cur[C::kLoads];
#pragma unroll
            for (int i = 0; i < C::kLoads; ++i)
                cur[i] = *reinterpret_cast<const uint4 *>(line + ((i ^ (ln & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            const int64_t g = ((blockIdx.x + lt * gridDim.x) * LINES) / kLinesPerGroup + warp * C::kGroupsPerWarp + gsub;
            quantize_lane<kF32, kSym>(cur, g, part, total_groups, qw, scales, zeros);
        }
    }
    __syncthreads();
}

}  // namespace w4
