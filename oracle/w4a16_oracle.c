/*
 * w4a16_oracle.c -- plain, slow, obviously-correct CPU oracle for group-wise
 * asymmetric INT4 weight-only quantization and the W4A16 matmul that consumes it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC (see oracle.py).
 * The fp32 steps below rely on IEEE binary32 arithmetic with round-to-nearest-even
 * (SSE on x86-64, no excess precision) and on rintf() under FE_TONEAREST, which
 * rounds halves to even.
 *
 * Where each step comes from (page titles of the source pages):
 *   - "From-Scratch INT4 Weight-Only Quantizer with Per-Group Scales and
 *     Zero-Points", section "Architecture Overview" (item 3: per-group min/max,
 *     scale = (max-min)/15, zero_point = round(-min/scale) clipped to [0,15]) and
 *     "Step 5"/"Step 6" (the min/max reduction and the scale/zero-point formulas).
 *   - "From Scratch: Building a GPTQ INT4 Quantizer in Pure Python", "Step 2"
 *     (q = clip(round(t/scale + zero_point), 0, 15)) and "Step 4"
 *     (dequantize = (q - zero_point) * scale).
 *   - "Build a GPTQ INT4 Quantization Engine in Python/NumPy", "Step 4" (two
 *     values per byte, column 2j in the low nibble, 2j+1 in the high nibble) and
 *     "Step 5" (the dequantize-matmul y = x @ W_dequant^T, computed over chunks
 *     of output rows so only a chunk of W is ever dequantized at once).
 *   - "Build a GPTQ INT4 Quantization Engine in Python/NumPy", "Step 3" (GPTQ:
 *     the columns are quantized left to right and each column's quantization
 *     error, divided by the diagonal of the Cholesky factor of H^-1, is fed into
 *     the columns not yet quantized).
 *   - "Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization with
 *     Per-Channel Scale", "Step 3" (per-token INT8 activations: s_a = max|A| / 127
 *     with max|A| clipped below at 1e-8, a_q = clip(round(A / s_a), -128, 127)) and
 *     "Step 5" (forward_quant: a_q * s_a times the dequantized INT4 weights).
 *   The fixed convention on top of those pages: groups are 128 contiguous
 *   elements along K of W[N,K]; scale in fp32 (1 if max == min); IEEE fp32
 *   division; round half to even; scales stored as fp16, zero-points as uint8;
 *   dequantization uses the stored fp16 scale.
 *
 *   - Symmetric variant: "Build a GPTQ INT4 Quantization Engine in Python/NumPy",
 *     "Step 2" (per-group absmax, scale = absmax / 7 with 1 for an all-zero group,
 *     q = clip(round(w / scale), -8, 7)); the group-wise INT4 layer page
 *     ("Building a From-Scratch Group-Wise INT4 Quantization Layer for LLaMA
 *     Weights", "Key design decisions") names symmetric per-group scales as the
 *     standard choice for transformer weights.
 *
 * Readings taken where the pages are silent or disagree:
 *   - q and zp are computed with the fp32 scale; only dequantization uses the
 *     stored fp16 scale.
 *   - q = clip(rint(w / s) + zp, 0, 15), i.e. rounding happens before adding zp
 *     (the pure-Python GPTQ page), not rint((w - min) / s).
 *   - Inputs are finite with a finite range; nothing here checks NaN/Inf.
 *   - Symmetric: groups along K as for the asymmetric format (the NumPy page groups
 *     output channels); the signed level q in [-8, 7] is stored as q + 8 with a zero
 *     point of 8, so (level - 8) * scale is the page's q * scale and the asymmetric
 *     layout and matmul apply unchanged.  The group-wise INT4 layer page's listing
 *     (scale = absmax, quantizing |w|) loses the sign and is not followed.
 *   - Dequantized output as a 16-bit tensor: the exact product (q - zp) * s16
 *     rounded once to nearest-even bfloat16 or binary16.
 *   - Clip-range calibration ("Building a From-Scratch Group-Wise INT4 Quantization
 *     Layer for LLaMA Weights", Step 4, ScaleCalibrator), per group of 128 along K:
 *       percentile: the clip range r is the p-th percentile of |w| with linear
 *         interpolation between order statistics, in fp32: h = fl(fl(p / 100) * 127),
 *         lo = floor(h), f = h - lo, r = a_lo + f * (a_lo+1 - a_lo) (two roundings);
 *         the step is s = r / 7 (1 when r == 0), as the absmax calibrator's range
 *         gives absmax / 7 (the page's listing divides by the range itself, which
 *         leaves only the levels -1, 0, 1 and is not followed).
 *       mse: the step itself is searched: candidates c_i = linspace(min|w|, max|w|, n)
 *         in fp32 (c_i = fl(min + fl(i * step)), step = fl((max - min) / (n - 1)),
 *         c_(n-1) = max exactly; n = 1 gives min); candidates below fl32(1e-10) are
 *         skipped; each is scored by mean((clamp(rint(w / c), -7, 7) * c - w)^2)
 *         summed in fp32 in index order, every product, difference and sum rounded
 *         once; the first candidate with the smallest score wins (strict <), and 1e-8
 *         when none is scored.
 *     Both store level clamp(rint(w / s), -7, 7) + 8 with zero point 8 (the page's
 *     [-7, 7] range) and the fp16-rounded step as the scale.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define ORACLE_GROUP 128

/* ---- IEEE binary16 <-> binary32, written from the format definition ---------
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal:    (-1)^s * 2^(e-15) * (1 + f/1024),   1 <= e <= 30
 * Subnormal: (-1)^s * 2^(-14)  * (f/1024),       e == 0
 * e == 31 is Inf/NaN (outside the oracle's contract, mapped to Inf/NaN anyway). */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);            /* f/1024 * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)f, e - 25); /* (1 + f/1024) * 2^(e-15) */
    if (sign) v = -v;
    return (float)v;                            /* exact: binary16 fits in binary32 */
}

/* Round a binary32 value to the nearest binary16, ties to even.  Done on the
 * exact real value: find the binary16 spacing (quantum) at |x|, divide, round
 * the quotient half-to-even with rint(), multiply back.  All double steps are
 * exact because |x| has at most 24 significant bits and the quantum is a power
 * of two. */
uint16_t oracle_f32_to_f16_bits(float xf)
{
    double x = (double)xf;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(a)) return 0x7e00;
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);                     /* a = m * 2^e2, m in [0.5,1) -> floor(log2 a) = e2-1 */
    int E = e2 - 1;
    if (E < -14) E = -14;              /* subnormal range shares the 2^-14 binade spacing */
    double quantum = ldexp(1.0, E - 10);
    double n = rint(a / quantum);      /* integer count of quanta, ties to even */
    double r = n * quantum;
    if (r >= 65520.0 || isinf(a))      /* 65520 = max finite + half ulp: rounds to Inf */
        return sign | 0x7c00;
    /* re-encode r, which is exactly representable in binary16 */
    if (r < ldexp(1.0, -14)) {
        return sign | (uint16_t)(r / ldexp(1.0, -24));
    }
    int er;
    double mr = frexp(r, &er);          /* r = mr * 2^er, mr in [0.5,1) */
    int ebits = (er - 1) + 15;
    uint16_t fbits = (uint16_t)((mr * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)(ebits << 10) | fbits;
}

/* Round a binary32 value to the nearest bfloat16, ties to even.  bfloat16 keeps the
 * sign, the 8 exponent bits and the top 7 fraction bits of binary32, so the result is
 * the high 16 bits, plus one when the dropped low 16 bits are above half an ulp
 * (0x8000), or exactly half with an odd kept pattern.  A carry out of the fraction
 * moves to the next binade (or to Inf), which is the correctly rounded value. */
uint16_t oracle_f32_to_bf16_bits(float xf)
{
    uint32_t u;
    memcpy(&u, &xf, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (uint16_t)((u >> 16) | 0x0040u);   /* NaN stays a quiet NaN */
    uint32_t hi = u >> 16, lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
    return (uint16_t)hi;
}

/* bfloat16 is the high half of a binary32 pattern: widening is a 16-bit shift. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- quantize one group ---------------------------------------------------- */
/* w: the group's values already widened (exactly) to binary32. */
static void quantize_group(const float *w, int G, uint8_t *q, float *scale, int *zero)
{
    /* min/max over the group (linear scan). */
    float mn = w[0], mx = w[0];
    for (int i = 1; i < G; ++i) {
        if (w[i] < mn) mn = w[i];
        if (w[i] > mx) mx = w[i];
    }
    /* scale = (max - min) / 15 in fp32; a constant group gets scale 1. */
    float s;
    if (mx == mn) {
        s = 1.0f;
    } else {
        float d = mx - mn;          /* fp32 subtraction */
        s = d / 15.0f;              /* IEEE fp32 division */
    }
    /* zero-point = clip(round_half_even(-min / scale), 0, 15); the clamp is done in
     * float so a huge quotient cannot overflow an int. */
    float negmn = -mn;
    float zq = rintf(negmn / s);
    float zc = fminf(fmaxf(zq, 0.0f), 15.0f);
    int zp = (int)zc;
    /* q = clip(round_half_even(w / scale) + zp, 0, 15). */
    for (int i = 0; i < G; ++i) {
        float t = rintf(w[i] / s) + (float)zp;
        float c = fminf(fmaxf(t, 0.0f), 15.0f);
        q[i] = (uint8_t)(int)c;
    }
    *scale = s;
    *zero = zp;
}

/* ---- quantize one group, symmetric ------------------------------------------ */
/* Page steps: absmax over the group, scale = absmax / 7 (IEEE fp32 division; 1 for
 * an all-zero group), q = clip(round_half_even(w / scale), -8, 7).  Stored level =
 * q + 8 with zero point 8. */
static void quantize_group_sym(const float *w, int G, uint8_t *q, float *scale, int *zero)
{
    float amax = 0.0f;
    for (int i = 0; i < G; ++i) {
        float a = fabsf(w[i]);
        if (a > amax) amax = a;
    }
    float s = (amax == 0.0f) ? 1.0f : amax / 7.0f;
    for (int i = 0; i < G; ++i) {
        float t = rintf(w[i] / s);
        float c = fminf(fmaxf(t, -8.0f), 7.0f);
        q[i] = (uint8_t)((int)c + 8);
    }
    *scale = s;
    *zero = 8;
}

/* ---- clip-range calibration ---------------------------------------------------- */
/* The page's symmetric level rule with the [-7, 7] range: level = q + 8. */
static void levels_sym7(const float *w, int G, float s, uint8_t *q)
{
    for (int i = 0; i < G; ++i) {
        float t = rintf(w[i] / s);
        float c = fminf(fmaxf(t, -7.0f), 7.0f);
        q[i] = (uint8_t)((int)c + 8);
    }
}

/* p-th percentile (0 < p <= 100) of |w| over the group, linear interpolation between
 * the order statistics (ascending a_0 <= ... <= a_(G-1)), in fp32. */
float oracle_percentile_abs(const float *w, int G, float p)
{
    float a[ORACLE_GROUP];
    for (int i = 0; i < G; ++i) a[i] = fabsf(w[i]);
    for (int i = 1; i < G; ++i) {           /* insertion sort, ascending */
        float v = a[i];
        int j = i - 1;
        while (j >= 0 && a[j] > v) {
            a[j + 1] = a[j];
            --j;
        }
        a[j + 1] = v;
    }
    float qf = p / 100.0f;
    float h = qf * (float)(G - 1);
    float fl = floorf(h);
    int lo = (int)fl;
    if (lo < 0) lo = 0;
    if (lo > G - 1) lo = G - 1;
    int hi = lo + 1 < G ? lo + 1 : G - 1;
    float f = h - fl;                       /* exact */
    float d = a[hi] - a[lo];
    float fd = f * d;
    return a[lo] + fd;
}

/* The step chosen by the MSE search over n candidates (see the header). */
float oracle_mse_step(const float *w, int G, int n)
{
    float lo = fabsf(w[0]), hi = lo;
    for (int i = 1; i < G; ++i) {
        float a = fabsf(w[i]);
        if (a < lo) lo = a;
        if (a > hi) hi = a;
    }
    const float thr = 1e-10f;
    float best_s = 1e-8f, best = INFINITY;
    float step = (n > 1) ? (hi - lo) / (float)(n - 1) : 0.0f;
    for (int i = 0; i < n; ++i) {
        float c;
        if (n == 1) c = lo;
        else if (i == n - 1) c = hi;
        else {
            float is = (float)i * step;
            c = lo + is;
        }
        if (c < thr) continue;
        float e = 0.0f;
        for (int k = 0; k < G; ++k) {
            float t = rintf(w[k] / c);
            t = fminf(fmaxf(t, -7.0f), 7.0f);
            float r = t * c;
            float d = r - w[k];
            float d2 = d * d;
            e = e + d2;
        }
        float mse = e / (float)G;
        if (mse < best) {
            best = mse;
            best_s = c;
        }
    }
    return best_s;
}

/* Calibrated symmetric quantization of one group: method 2 = percentile (param = p),
 * method 3 = MSE search (param = number of candidates). */
static void quantize_group_calib(const float *w, int G, int method, double param, uint8_t *q,
                                 float *scale, int *zero)
{
    float s;
    if (method == 2) {
        float r = oracle_percentile_abs(w, G, (float)param);
        s = (r == 0.0f) ? 1.0f : r / 7.0f;
    } else {
        s = oracle_mse_step(w, G, (int)param);
    }
    levels_sym7(w, G, s, q);
    *scale = s;
    *zero = 8;
}

/* Quantize and pack W[N,K] (row-major, K contiguous).
 *   w_dtype: 0 = fp16 bits (uint16), 1 = fp32
 *   qweight: uint8 [N, K/2], element 2j in the low nibble, 2j+1 in the high nibble
 *   scales : fp16 bits [N, K/128] (the fp32 scale rounded to nearest-even fp16)
 *   zeros  : uint8 [N, K/128]
 *   scales32 (optional, may be NULL): the fp32 scales, for tests of the bound.
 * Returns 0, or -1 on invalid arguments. */
static int quantize_pack_mode(const void *W, int w_dtype, int64_t N, int64_t K, int mode, double param,
                              uint8_t *qweight, uint16_t *scales, uint8_t *zeros, float *scales32)
{
    if (N < 0 || K < 0 || K % ORACLE_GROUP != 0) return -1;
    if (w_dtype != 0 && w_dtype != 1) return -1;
    const int64_t ng = K / ORACLE_GROUP;
    float wbuf[ORACLE_GROUP];
    uint8_t qbuf[ORACLE_GROUP];
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < ng; ++g) {
            const int64_t base = n * K + g * ORACLE_GROUP;
            for (int i = 0; i < ORACLE_GROUP; ++i) {
                if (w_dtype == 0)
                    wbuf[i] = oracle_f16_to_f32(((const uint16_t *)W)[base + i]);
                else
                    wbuf[i] = ((const float *)W)[base + i];
            }
            float s;
            int zp;
            if (mode == 1)
                quantize_group_sym(wbuf, ORACLE_GROUP, qbuf, &s, &zp);
            else if (mode >= 2)
                quantize_group_calib(wbuf, ORACLE_GROUP, mode, param, qbuf, &s, &zp);
            else
                quantize_group(wbuf, ORACLE_GROUP, qbuf, &s, &zp);
            scales[n * ng + g] = oracle_f32_to_f16_bits(s);
            zeros[n * ng + g] = (uint8_t)zp;
            if (scales32) scales32[n * ng + g] = s;
            for (int j = 0; j < ORACLE_GROUP / 2; ++j) {
                uint8_t lo = qbuf[2 * j], hi = qbuf[2 * j + 1];
                qweight[n * (K / 2) + g * (ORACLE_GROUP / 2) + j] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return 0;
}

int oracle_quantize_pack(const void *W, int w_dtype, int64_t N, int64_t K,
                         uint8_t *qweight, uint16_t *scales, uint8_t *zeros,
                         float *scales32)
{
    return quantize_pack_mode(W, w_dtype, N, K, 0, 0.0, qweight, scales, zeros, scales32);
}

/* The symmetric variant: same layouts, zero points all 8. */
int oracle_quantize_pack_sym(const void *W, int w_dtype, int64_t N, int64_t K,
                             uint8_t *qweight, uint16_t *scales, uint8_t *zeros,
                             float *scales32)
{
    return quantize_pack_mode(W, w_dtype, N, K, 1, 0.0, qweight, scales, zeros, scales32);
}

/* Clip-range calibrated symmetric variant: method 2 = percentile with p = param
 * (0 < p <= 100), method 3 = MSE search over (int)param >= 1 candidates. */
int oracle_quantize_pack_calib(const void *W, int w_dtype, int64_t N, int64_t K, int method,
                               double param, uint8_t *qweight, uint16_t *scales, uint8_t *zeros,
                               float *scales32)
{
    if (method == 2 && !(param > 0.0 && param <= 100.0)) return -1;
    if (method == 3 && !(param >= 1.0)) return -1;
    if (method != 2 && method != 3) return -1;
    return quantize_pack_mode(W, w_dtype, N, K, method, param, qweight, scales, zeros, scales32);
}

/* ---- GPTQ: second-order column-greedy quantization ------------------------------
 * "Build a GPTQ INT4 Quantization Engine in Python/NumPy", Step 3.  The page's listing
 * sweeps output rows with a K x K factor indexed by rows; the algorithm it names (and
 * follows in prose) sweeps the input columns, which is what is done here, row by row
 * (rows are independent):
 *   U = the upper-triangular Cholesky factor of H^-1 (H^-1 = U^T U), given as fp32 [K,K]
 *       (computed by the caller from the calibration activations).
 *   w = the row, widened exactly to fp32.  For j = 0 .. K-1:
 *     at a group start (j % 128 == 0): the group's s and zp from the current values
 *       w[j .. j+127] by the rule of w4_quantize_pack (fp32 min/max, s = (max-min)/15
 *       or 1, zp = clip(rint(-min/s), 0, 15)), s16 = fp16(s);
 *     q_j = clip(rint(w_j / s) + zp, 0, 15);
 *     e   = (w_j - (q_j - zp) * s16) / U[j][j]        (the reconstruction inference uses)
 *     w_c = fmaf(-e, U[j][c], w_c) for c = j+1 .. K-1, in that order.
 * Every operation is IEEE fp32 with round-to-nearest-even (fmaf fused).  Outputs in
 * the layout of oracle_quantize_pack. */
int oracle_gptq_quantize(const void *W, int w_dtype, int64_t N, int64_t K, const float *U,
                         uint8_t *qweight, uint16_t *scales, uint8_t *zeros)
{
    if (N < 0 || K < 0 || K % ORACLE_GROUP != 0) return -1;
    if (w_dtype != 0 && w_dtype != 1) return -1;
    const int64_t ng = K / ORACLE_GROUP;
    float *w = (float *)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
    uint8_t *q = (uint8_t *)malloc((size_t)(K > 0 ? K : 1));
    if (!w || !q) { free(w); free(q); return -2; }
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k)
            w[k] = (w_dtype == 0) ? oracle_f16_to_f32(((const uint16_t *)W)[n * K + k])
                                  : ((const float *)W)[n * K + k];
        float s = 1.0f, s16f = 1.0f;
        int zp = 0;
        for (int64_t j = 0; j < K; ++j) {
            if (j % ORACLE_GROUP == 0) {
                uint8_t scratch[ORACLE_GROUP];
                quantize_group(w + j, ORACLE_GROUP, scratch, &s, &zp);
                uint16_t sb = oracle_f32_to_f16_bits(s);
                s16f = oracle_f16_to_f32(sb);
                scales[n * ng + j / ORACLE_GROUP] = sb;
                zeros[n * ng + j / ORACLE_GROUP] = (uint8_t)zp;
            }
            float t = rintf(w[j] / s) + (float)zp;
            float c = fminf(fmaxf(t, 0.0f), 15.0f);
            q[j] = (uint8_t)(int)c;
            float rec = (float)((int)q[j] - zp) * s16f;
            float d = w[j] - rec;
            float e = d / U[j * K + j];
            for (int64_t cc = j + 1; cc < K; ++cc)
                w[cc] = fmaf(-e, U[j * K + cc], w[cc]);
        }
        for (int64_t jb = 0; jb < K / 2; ++jb)
            qweight[n * (K / 2) + jb] = (uint8_t)(q[2 * jb] | (q[2 * jb + 1] << 4));
    }
    free(w);
    free(q);
    return 0;
}

/* Unpack qweight[N,K/2] into q[N,K] (one value 0..15 per byte). */
int oracle_unpack(const uint8_t *qweight, int64_t N, int64_t K, uint8_t *q)
{
    if (N < 0 || K < 0 || K % 2 != 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 2; ++j) {
            uint8_t b = qweight[n * (K / 2) + j];
            q[n * K + 2 * j] = b & 0x0f;
            q[n * K + 2 * j + 1] = (b >> 4) & 0x0f;
        }
    return 0;
}

/* Dequantize rows [n0, n0+rows) into out[rows, K] in fp64:
 * w_hat[n,k] = (q[n,k] - zp[n,k/128]) * fp16_scale[n,k/128]  (exact in fp64). */
static void dequant_rows(const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                         int64_t n0, int64_t rows, int64_t K, double *out)
{
    const int64_t ng = K / ORACLE_GROUP;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t n = n0 + r;
        for (int64_t k = 0; k < K; ++k) {
            uint8_t b = qweight[n * (K / 2) + k / 2];
            int q = (k & 1) ? (b >> 4) & 0x0f : b & 0x0f;
            int64_t g = k / ORACLE_GROUP;
            double s = (double)oracle_f16_to_f32(scales[n * ng + g]);
            int zp = zeros[n * ng + g];
            out[r * K + k] = (double)(q - zp) * s;
        }
    }
}

int oracle_dequantize(const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                      int64_t N, int64_t K, double *W_hat)
{
    if (N < 0 || K < 0 || K % ORACLE_GROUP != 0) return -1;
    dequant_rows(qweight, scales, zeros, 0, N, K, W_hat);
    return 0;
}

/* Dequantize into a 16-bit tensor: out[n,k] = RNE((q - zp) * s16), out_dtype 0 =
 * bfloat16, 1 = binary16 (bit patterns).  The fp64 product is exact and also exact in
 * binary32 (a 5-bit integer times an 11-bit significand), so it is narrowed to
 * binary32 without rounding and then rounded once. */
int oracle_dequantize_16(const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                         int64_t N, int64_t K, int out_dtype, uint16_t *out)
{
    if (N < 0 || K < 0 || K % ORACLE_GROUP != 0) return -1;
    if (out_dtype != 0 && out_dtype != 1) return -1;
    double row[ORACLE_GROUP];
    const int64_t ng = K / ORACLE_GROUP;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < ng; ++g) {
            for (int i = 0; i < ORACLE_GROUP; ++i) {
                int64_t k = g * ORACLE_GROUP + i;
                uint8_t b = qweight[n * (K / 2) + k / 2];
                int q = (k & 1) ? (b >> 4) & 0x0f : b & 0x0f;
                double s = (double)oracle_f16_to_f32(scales[n * ng + g]);
                row[i] = (double)(q - zeros[n * ng + g]) * s;
            }
            for (int i = 0; i < ORACLE_GROUP; ++i) {
                float f = (float)row[i];
                if ((double)f != row[i]) return -2;   /* cannot happen; see above */
                out[n * K + g * ORACLE_GROUP + i] =
                    out_dtype == 0 ? oracle_f32_to_bf16_bits(f) : oracle_f32_to_f16_bits(f);
            }
        }
    return 0;
}

/* W4A16 matmul in fp64:  Y[m,n] = sum_k A[m,k] * w_hat[n,k]   (A bf16 [M,K])
 * and S[m,n] = sum_k |A[m,k] * w_hat[n,k]| (the scale of the tolerance).
 * Follows the chunked dequantize-matmul pattern: dequantize a chunk of output rows,
 * then take the dot products against every activation row. */
/* Y = a * W_hat^T and S = sum |a * w_hat| in fp64 for activations already in fp64,
 * over chunks of 256 output rows ([P4] Step 5's chunked dequantize-matmul). */
static int matmul_f64(const double *a, int64_t M, int64_t N, int64_t K,
                      const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                      double *Y, double *S)
{
    const int64_t chunk = 256;
    double *wc = (double *)malloc(sizeof(double) * (size_t)(chunk * K > 0 ? chunk * K : 1));
    if (!wc) return -2;
    for (int64_t n0 = 0; n0 < N; n0 += chunk) {
        int64_t rows = (N - n0 < chunk) ? N - n0 : chunk;
        dequant_rows(qweight, scales, zeros, n0, rows, K, wc);
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t r = 0; r < rows; ++r) {
                double acc = 0.0, sab = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double p = a[m * K + k] * wc[r * K + k];
                    acc += p;
                    sab += fabs(p);
                }
                Y[m * N + n0 + r] = acc;
                if (S) S[m * N + n0 + r] = sab;
            }
        }
    }
    free(wc);
    return 0;
}

int oracle_matmul(const uint16_t *A, int64_t M, int64_t N, int64_t K,
                  const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                  double *Y, double *S)
{
    if (M < 0 || N < 0 || K < 0 || K % ORACLE_GROUP != 0) return -1;
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!a) return -2;
    for (int64_t i = 0; i < M * K; ++i) a[i] = oracle_bf16_to_f64(A[i]);
    int rc = matmul_f64(a, M, N, K, qweight, scales, zeros, Y, S);
    free(a);
    return rc;
}

/* ---- W4A8: per-token INT8 dynamic activation quantization -------------------------
 * "Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization with Per-Channel
 * Scale", Step 3 (activations_to_int8): per token (row of A), in fp32,
 *     s_a = max(max_k |a|, 1e-8) / 127,   a_q = clip(round_half_even(a / s_a), -128, 127).
 * A arrives as bf16 (the library's activation type) and widens exactly to fp32. */
int oracle_quantize_act_int8(const uint16_t *A, int64_t M, int64_t K, int8_t *a_q, float *a_scale)
{
    if (M < 0 || K < 0) return -1;
    for (int64_t m = 0; m < M; ++m) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = fabsf((float)oracle_bf16_to_f64(A[m * K + k]));
            if (v > amax) amax = v;
        }
        float s = fmaxf(amax, 1e-8f) / 127.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = (float)oracle_bf16_to_f64(A[m * K + k]);
            float t = rintf(v / s);
            t = fminf(fmaxf(t, -128.0f), 127.0f);
            a_q[m * K + k] = (int8_t)(int)t;
        }
        a_scale[m] = s;
    }
    return 0;
}

/* The W4A8 product (Step 5, forward_quant: the INT8 activations times their per-token
 * scale, multiplied by the dequantized INT4 weights), in fp64:
 *     Y[m,n] = sum_k (a_q[m,k] * s_a[m]) * w_hat[n,k],  S = sum_k |...|.
 * Every product is exact in fp64 (8 + 24 + 4 + 11 significant bits). */
int oracle_w4a8_matmul(const int8_t *a_q, const float *a_scale, int64_t M, int64_t N, int64_t K,
                       const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                       double *Y, double *S)
{
    if (M < 0 || N < 0 || K < 0 || K % ORACLE_GROUP != 0) return -1;
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!a) return -2;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            a[m * K + k] = (double)a_q[m * K + k] * (double)a_scale[m];
    int rc = matmul_f64(a, M, N, K, qweight, scales, zeros, Y, S);
    free(a);
    return rc;
}

/* The W4A8 product for a list of (m, n) output positions, one by one (checks of
 * full-size outputs on a sample): Y = sum_k (a_q[m,k] * s_a[m]) * w_hat[n,k] in fp64. */
int oracle_w4a8_matmul_entries(const int8_t *a_q, const float *a_scale, int64_t M, int64_t N, int64_t K,
                               const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                               const int64_t *mi, const int64_t *ni, int64_t count, double *Y, double *S)
{
    if (M < 0 || N < 0 || K < 0 || K % ORACLE_GROUP != 0) return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!w) return -2;
    for (int64_t t = 0; t < count; ++t) {
        int64_t m = mi[t], n = ni[t];
        if (m < 0 || m >= M || n < 0 || n >= N) { free(w); return -1; }
        dequant_rows(qweight, scales, zeros, n, 1, K, w);
        double acc = 0.0, sab = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = ((double)a_q[m * K + k] * (double)a_scale[m]) * w[k];
            acc += p;
            sab += fabs(p);
        }
        Y[t] = acc;
        if (S) S[t] = sab;
    }
    free(w);
    return 0;
}

/* The same quantity for a list of (m, n) output positions, one by one; used to
 * check full-size outputs on a sample. */
int oracle_matmul_entries(const uint16_t *A, int64_t M, int64_t N, int64_t K,
                          const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                          const int64_t *mi, const int64_t *ni, int64_t count,
                          double *Y, double *S)
{
    if (M < 0 || N < 0 || K < 0 || K % ORACLE_GROUP != 0) return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!w) return -2;
    for (int64_t t = 0; t < count; ++t) {
        int64_t m = mi[t], n = ni[t];
        if (m < 0 || m >= M || n < 0 || n >= N) { free(w); return -1; }
        dequant_rows(qweight, scales, zeros, n, 1, K, w);
        double acc = 0.0, sab = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = oracle_bf16_to_f64(A[m * K + k]) * w[k];
            acc += p;
            sab += fabs(p);
        }
        Y[t] = acc;
        if (S) S[t] = sab;
    }
    free(w);
    return 0;
}
