// w4a16_api.cu -- the extern "C" entry points of libw4a16 (see include/w4a16.h).
//
// One translation unit holds every kernel, so the device error word is a single
// symbol.  The entry points validate arguments on the host, pick a kernel, and
// enqueue it on the caller's stream with cudaLaunchKernelEx (whose return value is
// the launch status); they never synchronize and never allocate.
#include <atomic>
#include <cmath>
#include <map>
#include <mutex>
#include <utility>

#include "act_quant.cuh"
#include "common.cuh"
#include "dequantize.cuh"
#include "gemm_tcgen05.cuh"
#include "gemv.cuh"
#include "gemv_dp4a.cuh"
#include "gemv_mma.cuh"
#include "gptq.cuh"
#include "quantize_calib.cuh"
#include "quantize_pack.cuh"

// Scratch of w4_matmul_w4a8_noalloc: a fixed device array, part of the library's image
// on every GPU that loads it (held until the process exits), so that entry point never
// allocates.  Host code must not pass its name to a kernel: the name is a host-side
// stand-in; the device address comes from cudaGetSymbolAddress (noalloc_scratch below).
static __device__ __align__(256) uint8_t g_w4a8_noalloc_scratch[W4_NOALLOC_SCRATCH_BYTES];

namespace {

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_stall{0};

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    std::once_flag once;
    int sm_count = 0;
    cudaError_t err = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];

// Number of SMs of the current device (cached per device).
int current_sm_count(int *sm_count) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W4_ERR_CUDA;
    DeviceInfo &d = g_dev[dev];
    std::call_once(d.once, [&]() {
        d.err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    });
    if (d.err != cudaSuccess || d.sm_count <= 0) return W4_ERR_CUDA;
    *sm_count = d.sm_count;
    return W4_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Device address of the no-allocation scratch array on the current device, looked up
// once per device (with that device current) and cached.
struct ScratchAddr {
    std::once_flag once;
    void *ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
ScratchAddr g_scratch_addr[kMaxDevices];

int noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W4_ERR_CUDA;
    ScratchAddr &sa = g_scratch_addr[dev];
    std::call_once(sa.once, [&]() { sa.err = cudaGetSymbolAddress(&sa.ptr, g_w4a8_noalloc_scratch); });
    if (sa.err != cudaSuccess || sa.ptr == nullptr) return W4_ERR_CUDA;
    *out = sa.ptr;
    return W4_OK;
}

w4::WaitParams wait_params() {
    w4::WaitParams w;
    w.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    w.stall = g_stall.load(std::memory_order_relaxed);
    return w;
}

template <typename Kern, typename... Args>
int launch(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

// As launch(), with programmatic dependent launch: the kernel may begin launching while
// the previous kernel in the stream finishes; it must execute griddepcontrol.wait before
// touching global memory.
template <typename Kern, typename... Args>
int launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

// Raises a kernel's dynamic shared-memory limit once per device (and per size).
int ensure_smem_attr(const void *kernel, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    int &have = done[{dev, kernel}];
    if (have >= bytes) return W4_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return W4_ERR_CUDA;
    have = bytes;
    return W4_OK;
}

template <typename Kern>
int launch_gemv_kernel(Kern kern, int threads, const CUtensorMap &tmS, const CUtensorMap &tmZ,
                       const w4::gemv::Params &prm, int64_t grid, size_t smem, cudaStream_t stream) {
    if (int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), static_cast<int>(smem))) return rc;
    return launch(kern, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, stream, tmS, tmZ, prm);
}

int launch_gemv_simple(const __nv_bfloat16 *A, int64_t M, int64_t N, int64_t K, const uint8_t *qweight,
                       const __half *scales, const uint8_t *zeros, __nv_bfloat16 *Y,
                       cudaStream_t stream, int sms) {
    constexpr int R = 2;
    const int64_t warps_needed = (N + R - 1) / R;
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    switch (M) {
        case 1: return launch(w4::gemv_simple_kernel<1, R>, grid, block, 0, stream, A, qweight, scales, zeros, Y, N, K);
        case 2: return launch(w4::gemv_simple_kernel<2, R>, grid, block, 0, stream, A, qweight, scales, zeros, Y, N, K);
        case 3: return launch(w4::gemv_simple_kernel<3, R>, grid, block, 0, stream, A, qweight, scales, zeros, Y, N, K);
        case 4: return launch(w4::gemv_simple_kernel<4, R>, grid, block, 0, stream, A, qweight, scales, zeros, Y, N, K);
        case 5: return launch(w4::gemv_simple_kernel<5, R>, grid, block, 0, stream, A, qweight, scales, zeros, Y, N, K);
        case 6: return launch(w4::gemv_simple_kernel<6, R>, grid, block, 0, stream, A, qweight, scales, zeros, Y, N, K);
        case 7: return launch(w4::gemv_simple_kernel<7, R>, grid, block, 0, stream, A, qweight, scales, zeros, Y, N, K);
        case 8: return launch(w4::gemv_simple_kernel<8, R>, grid, block, 0, stream, A, qweight, scales, zeros, Y, N, K);
        default: return W4_ERR_INVALID_ARG;
    }
}

constexpr size_t kGemvSmemLimit = 220 * 1024;

// M = 1 on integer dot products: K a multiple of 2048 up to 16384, 16-byte aligned
// scales and zero points.  Returns W4_ERR_UNSUPPORTED for other shapes.
int launch_gemv_dp4a(const void *A, bool i8, const float *row_scale, int64_t N, int64_t K, const uint8_t *qweight,
                     const __half *scales, const uint8_t *zeros, __nv_bfloat16 *Y, cudaStream_t stream,
                     int sms, w4::WaitParams wp) {
    namespace gd = w4::gemv_dp4a;
    if (K % 2048 != 0 || K > 16384 || !aligned(scales, 16) || !aligned(zeros, 16) || N > INT32_MAX / 2)
        return W4_ERR_UNSUPPORTED;
    const int k = static_cast<int>(K), ng = k / 128;
    // A lane owns a 128-group (half of one when K = 2048); WR warps share a row, WR
    // the smallest divisor of the consumer-warp count covering the row's pieces.
    const int H = ng >= 32 ? 1 : 2;
    int WR = 1;
    while (WR <= gd::CW && (32 * WR < H * ng || gd::CW % WR != 0)) ++WR;
    if (WR > gd::CW) return W4_ERR_UNSUPPORTED;
    // The conversion's per-segment maxima (K / 16 words) borrow the reduction ring.
    if (static_cast<int64_t>(gd::RS) * (gd::CW / WR) * gd::RB * (32 * WR + 1) < k / 16) return W4_ERR_UNSUPPORTED;
    int stages = 0, smem = 0;
    for (int s = gd::MAX_STAGES; s >= 2; --s) {
        const int total = H == 1 ? gd::Layout<1>(k, WR, s).total : gd::Layout<2>(k, WR, s).total;
        if (total <= gd::SMEM_LIMIT) {
            stages = s;
            smem = total;
            break;
        }
    }
    if (stages == 0) return W4_ERR_UNSUPPORTED;
    gd::Params prm;
    prm.A = A;
    prm.row_scale = row_scale;
    prm.qweight = qweight;
    prm.scales = scales;
    prm.zeros = zeros;
    prm.Y = Y;
    prm.N = static_cast<int>(N);
    prm.K = k;
    prm.WR = WR;
    prm.stages = stages;
    prm.wait = wp;
    int64_t grid = N < sms ? N : sms;
    const int64_t per_cta = (N + grid - 1) / grid;
    grid = (N + per_cta - 1) / per_cta;
    prm.rows_per_cta = static_cast<int>(per_cta);
    auto kern = H == 1 ? (i8 ? gd::w4a16_gemv_dp4a_kernel<1, true> : gd::w4a16_gemv_dp4a_kernel<1, false>)
                       : (i8 ? gd::w4a16_gemv_dp4a_kernel<2, true> : gd::w4a16_gemv_dp4a_kernel<2, false>);
    if (int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem)) return rc;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(gd::NUM_THREADS), smem, stream, prm);
}

// 1 <= M <= 16 on warp-level tensor-core MMAs with the weights dequantized in
// registers: K a multiple of 2048, the activations (M x K bf16 after widening) resident
// in shared memory next to at least two stages.  Scale and zero-point tables must be
// 16-byte aligned (W4_ERR_MISALIGNED otherwise when `strict`, else UNSUPPORTED so the
// caller can pick another kernel).  Returns W4_ERR_UNSUPPORTED for other shapes.
// A is bf16, or int8 when i8 (W4A8); row_scale (may be null) multiplies output row m.
bool gemv_mma_shape_ok(int64_t M, int64_t K) {
    namespace gm = w4::gmma;
    if (M < 1 || M > 16 || K % gm::k_per_stage(1) != 0 || K > (int64_t(1) << 20)) return false;
    int gpw = 0, stages = 0;
    gm::plan(static_cast<int>(M), static_cast<int>(K), &gpw, &stages);
    return stages > 0;
}

int launch_gemv_mma(const void *A, bool i8, const float *row_scale, int64_t M, int64_t N, int64_t K,
                    const uint8_t *qweight, const __half *scales, const uint8_t *zeros, __nv_bfloat16 *Y,
                    cudaStream_t stream, int sms, w4::WaitParams wp, bool strict) {
    namespace gm = w4::gmma;
    if (!gemv_mma_shape_ok(M, K) || N > INT32_MAX / 2) return W4_ERR_UNSUPPORTED;
    if (!aligned(scales, 16) || !aligned(zeros, 16)) return strict ? W4_ERR_MISALIGNED : W4_ERR_UNSUPPORTED;
    const int m = static_cast<int>(M), k = static_cast<int>(K);
    const int nb = m <= 8 ? 1 : 2;
    int gpw = 0, stages = 0;
    gm::plan(m, k, &gpw, &stages);
    const bool regb = gm::regb_ok(m, k, gpw);
    const int smem = gm::smem_bytes(m, k, nb, gpw, stages, regb);
    gm::Params prm;
    prm.A = A;
    prm.qweight = qweight;
    prm.scales = scales;
    prm.zeros = zeros;
    prm.row_scale = row_scale;
    prm.Y = Y;
    prm.M = m;
    prm.N = static_cast<int>(N);
    prm.K = k;
    prm.tiles = static_cast<int>((N + gm::ROWS - 1) / gm::ROWS);
    prm.stages = stages;
    prm.wait = wp;
    const int grid = prm.tiles < sms ? prm.tiles : sms;
    CUtensorMap tmW, tmS, tmZ;
    if (!gm::make_maps(&tmW, &tmS, &tmZ, qweight, scales, zeros, N, K, gpw)) return W4_ERR_CUDA;
    decltype(&gm::gemv_mma_kernel<1, 1, false, false>) kern;
    if (regb && gpw == 2) kern = i8 ? gm::gemv_mma_kernel<1, 2, true, true> : gm::gemv_mma_kernel<1, 2, false, true>;
    else if (regb) kern = i8 ? gm::gemv_mma_kernel<1, 1, true, true> : gm::gemv_mma_kernel<1, 1, false, true>;
    else if (nb == 1 && gpw == 2)
        kern = i8 ? gm::gemv_mma_kernel<1, 2, true, false> : gm::gemv_mma_kernel<1, 2, false, false>;
    else if (nb == 1) kern = i8 ? gm::gemv_mma_kernel<1, 1, true, false> : gm::gemv_mma_kernel<1, 1, false, false>;
    else kern = i8 ? gm::gemv_mma_kernel<2, 1, true, false> : gm::gemv_mma_kernel<2, 1, false, false>;
    if (int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem)) return rc;
    return launch_pdl(kern, dim3(grid), dim3(gm::NUM_THREADS), smem, stream, tmW, tmS, tmZ, prm);
}

// M <= 8.  The streaming kernels need the scales / zero points reachable by 2-D tensor
// copies (K a multiple of 2048, 16-byte aligned tables, K <= 32768); otherwise the
// plain kernel runs.  Activations in registers when M * ceil(K / 4096) <= 2, in shared
// memory otherwise (if they fit).
int launch_gemv(const __nv_bfloat16 *A, int64_t M, int64_t N, int64_t K, const uint8_t *qweight,
                const __half *scales, const uint8_t *zeros, __nv_bfloat16 *Y,
                cudaStream_t stream, int sms, w4::WaitParams wp) {
    namespace gv = w4::gemv;
    if (M == 1) {
        const int rc = launch_gemv_dp4a(A, false, nullptr, N, K, qweight, scales, zeros, Y, stream, sms, wp);
        if (rc != W4_ERR_UNSUPPORTED) return rc;
    }
    const int64_t ng = K / 128;
    const bool tma_ok = (K % 2048 == 0) && K <= 32768 && aligned(scales, 16) && aligned(zeros, 16) &&
                        N <= INT32_MAX / 2;
    const int64_t gpl = (ng + 31) / 32;
    const bool rega = tma_ok && M * gpl <= 2;
    // 16 consumer warps when a lane's activations take 64 registers, 8 when 128.
    const int cw = (rega && M * gpl == 1) ? gv::CW_REGA : gv::CW_SMEMA;
    size_t smem = kGemvSmemLimit + 1;
    int stages = 0;
    if (tma_ok) {
        const int64_t sb = gv::stage_bytes(static_cast<int>(K), cw);
        stages = static_cast<int>(gv::RING_BYTES / sb);
        if (stages > gv::MAX_STAGES) stages = gv::MAX_STAGES;
        if (!rega) {
            const size_t fixed = gv::smem_bytes_smema(static_cast<int>(M), static_cast<int>(K), 0);
            const int64_t room = static_cast<int64_t>(kGemvSmemLimit) - static_cast<int64_t>(fixed);
            if (stages > room / sb) stages = static_cast<int>(room / sb);
        }
        if (stages >= 2)
            smem = rega ? gv::smem_bytes_rega(static_cast<int>(K), stages, cw)
                        : gv::smem_bytes_smema(static_cast<int>(M), static_cast<int>(K), stages);
    }
    if (!tma_ok || stages < 2 || smem > kGemvSmemLimit)
        return launch_gemv_simple(A, M, N, K, qweight, scales, zeros, Y, stream, sms);

    CUtensorMap tmS, tmZ;
    if (!w4::gemm::make_map_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, ng, N, ng * 2,
                               static_cast<uint32_t>(ng), cw, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !w4::gemm::make_map_2d(&tmZ, CU_TENSOR_MAP_DATA_TYPE_UINT8, zeros, ng, N, ng,
                               static_cast<uint32_t>(ng), cw, CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4_ERR_CUDA;

    // Contiguous bands of rows, at most one CTA per SM.
    int64_t grid = (N + cw - 1) / cw;
    if (grid > sms) grid = sms;
    const int64_t per_cta = (N + grid - 1) / grid;
    grid = (N + per_cta - 1) / per_cta;

    gv::Params prm;
    prm.A = A;
    prm.qweight = qweight;
    prm.Y = Y;
    prm.N = static_cast<int>(N);
    prm.K = static_cast<int>(K);
    prm.rows_per_cta = static_cast<int>(per_cta);
    prm.stages = stages;
    prm.wait = wp;
    const int tr = gv::num_threads(gv::CW_REGA), ts = gv::num_threads(gv::CW_SMEMA);
    if (rega) {
        if (M == 1 && gpl == 1) return launch_gemv_kernel(gv::gemv_rega_kernel<1, 1, gv::CW_REGA>, tr, tmS, tmZ, prm, grid, smem, stream);
        if (M == 1 && gpl == 2) return launch_gemv_kernel(gv::gemv_rega_kernel<1, 2, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        if (M == 2 && gpl == 1) return launch_gemv_kernel(gv::gemv_rega_kernel<2, 1, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
    }
    switch (M) {
        case 1: return launch_gemv_kernel(gv::gemv_smema_kernel<1, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        case 2: return launch_gemv_kernel(gv::gemv_smema_kernel<2, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        case 3: return launch_gemv_kernel(gv::gemv_smema_kernel<3, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        case 4: return launch_gemv_kernel(gv::gemv_smema_kernel<4, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        case 5: return launch_gemv_kernel(gv::gemv_smema_kernel<5, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        case 6: return launch_gemv_kernel(gv::gemv_smema_kernel<6, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        case 7: return launch_gemv_kernel(gv::gemv_smema_kernel<7, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        case 8: return launch_gemv_kernel(gv::gemv_smema_kernel<8, gv::CW_SMEMA>, ts, tmS, tmZ, prm, grid, smem, stream);
        default: return W4_ERR_INVALID_ARG;
    }
}

// Both quantizers: validation, the tensor map of W and the launch.
template <bool kSym>
int quantize_pack_impl(const void *W, int w_dtype, int64_t N, int64_t K, int group, uint8_t *qweight,
                       void *scales, uint8_t *zeros, cudaStream_t stream) {
    if (N < 0 || K < 0 || group <= 0) return W4_ERR_INVALID_ARG;
    if (w_dtype != W4_DTYPE_F16 && w_dtype != W4_DTYPE_F32) return W4_ERR_INVALID_ARG;
    if (group != W4_GROUP_SIZE) return W4_ERR_UNSUPPORTED;
    if (K % group != 0) return W4_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return W4_OK;
    if (!W || !qweight || !scales || !zeros) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(qweight, 16) || !aligned(scales, 2)) return W4_ERR_MISALIGNED;
    int sms = 0;
    if (int rc = current_sm_count(&sms)) return rc;

    const int64_t total_groups = N * (K / W4_GROUP_SIZE);
    uint32_t *qw = reinterpret_cast<uint32_t *>(qweight);
    __half *sc = static_cast<__half *>(scales);
    // W as bytes in 128-byte lines (2 per fp16 group, 4 per fp32 group), streamed by
    // 128 x 256-line tensor copies with 128-byte swizzle.
    const int lines_per_group = w_dtype == W4_DTYPE_F16 ? 2 : 4;
    const int64_t total_lines = total_groups * lines_per_group;
    if (total_lines >= (int64_t(1) << 31)) return W4_ERR_UNSUPPORTED;
    CUtensorMap tmW;
    if (!w4::gemm::make_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, 128, static_cast<uint64_t>(total_lines), 128,
                               128, w4::quant::BOX_LINES, CU_TENSOR_MAP_SWIZZLE_128B))
        return W4_ERR_CUDA;
    const int64_t units = (total_lines + w4::quant::LINES - 1) / w4::quant::LINES;
    const dim3 grid(static_cast<unsigned>(units < sms ? units : sms));
    const dim3 block(w4::quant::NUM_THREADS);
    const w4::WaitParams wp = wait_params();
    if (w_dtype == W4_DTYPE_F16) {
        auto kern = w4::quantize_pack_kernel<false, kSym>;
        if (int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), w4::quant::SMEM_BYTES)) return rc;
        return launch_pdl(kern, grid, block, w4::quant::SMEM_BYTES, stream, tmW, total_groups, qw, sc, zeros, wp,
                          static_cast<const uint8_t *>(W));
    }
    auto kern = w4::quantize_pack_kernel<true, kSym>;
    if (int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), w4::quant::SMEM_BYTES)) return rc;
    return launch_pdl(kern, grid, block, w4::quant::SMEM_BYTES, stream, tmW, total_groups, qw, sc, zeros, wp,
                      static_cast<const uint8_t *>(W));
}

// Both calibrated quantizers: validation and the launch (one warp per group; one thread
// per group for percentiles within 8 of either end of the group).
int quantize_calib_impl(bool mse, const void *W, int w_dtype, int64_t N, int64_t K, int group, float pct,
                        int candidates, uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream) {
    if (N < 0 || K < 0 || group <= 0) return W4_ERR_INVALID_ARG;
    if (w_dtype != W4_DTYPE_F16 && w_dtype != W4_DTYPE_F32) return W4_ERR_INVALID_ARG;
    if (mse ? (candidates < 1 || candidates > (1 << 24)) : !(pct > 0.0f && pct <= 100.0f))
        return W4_ERR_INVALID_ARG;
    if (group != W4_GROUP_SIZE) return W4_ERR_UNSUPPORTED;
    if (K % group != 0) return W4_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return W4_OK;
    if (!W || !qweight || !scales || !zeros) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(qweight, 16) || !aligned(scales, 2)) return W4_ERR_MISALIGNED;
    if (N > INT64_MAX / K) return W4_ERR_INVALID_ARG;
    int sms = 0;
    if (int rc = current_sm_count(&sms)) return rc;
    namespace cb = w4::calib;
    cb::Params prm;
    prm.W = W;
    prm.groups = N * (K / W4_GROUP_SIZE);
    prm.qweight = qweight;
    prm.scales = static_cast<__half *>(scales);
    prm.zeros = zeros;
    prm.p = pct;
    prm.n = candidates;
    int64_t blocks = (prm.groups + cb::WARPS - 1) / cb::WARPS;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid(static_cast<unsigned>(blocks)), block(cb::NUM_THREADS);
    const bool f32 = w_dtype == W4_DTYPE_F32;
    if (mse)
        return f32 ? launch(cb::calib_mse_kernel<true>, grid, block, 0, stream, prm)
                   : launch(cb::calib_mse_kernel<false>, grid, block, 0, stream, prm);
    // The order statistics the percentile needs (same fp32 arithmetic as the kernels):
    // within 8 of either end of the group, one thread per group keeps a short sorted list.
    const float qf = pct / 100.0f;
    const float h = qf * 127.0f;
    const int fl = static_cast<int>(std::floor(h));
    const int lo = fl < 0 ? 0 : (fl > 127 ? 127 : fl);
    const int hi = lo + 1 < 127 ? lo + 1 : 127;
    if (lo >= 120 || hi <= 7) {
        int64_t tblocks = (prm.groups + cb::NUM_THREADS - 1) / cb::NUM_THREADS;
        if (tblocks > cap) tblocks = cap;
        const dim3 tgrid(static_cast<unsigned>(tblocks));
        const bool top = lo >= 120, two = top ? lo >= 126 : hi <= 1;
        if (top && two)
            return f32 ? launch(cb::calib_percentile_ends_kernel<true, true, 2>, tgrid, block, 0, stream, prm)
                       : launch(cb::calib_percentile_ends_kernel<false, true, 2>, tgrid, block, 0, stream, prm);
        if (top)
            return f32 ? launch(cb::calib_percentile_ends_kernel<true, true, 8>, tgrid, block, 0, stream, prm)
                       : launch(cb::calib_percentile_ends_kernel<false, true, 8>, tgrid, block, 0, stream, prm);
        if (two)
            return f32 ? launch(cb::calib_percentile_ends_kernel<true, false, 2>, tgrid, block, 0, stream, prm)
                       : launch(cb::calib_percentile_ends_kernel<false, false, 2>, tgrid, block, 0, stream, prm);
        return f32 ? launch(cb::calib_percentile_ends_kernel<true, false, 8>, tgrid, block, 0, stream, prm)
                   : launch(cb::calib_percentile_ends_kernel<false, false, 8>, tgrid, block, 0, stream, prm);
    }
    return f32 ? launch(cb::calib_percentile_kernel<true>, grid, block, 0, stream, prm)
               : launch(cb::calib_percentile_kernel<false>, grid, block, 0, stream, prm);
}

}  // namespace

extern "C" {

const char *w4_status_string(int status) {
    switch (status) {
        case W4_OK: return "W4_OK";
        case W4_ERR_INVALID_ARG: return "W4_ERR_INVALID_ARG: invalid argument";
        case W4_ERR_UNSUPPORTED: return "W4_ERR_UNSUPPORTED: unsupported configuration (group must be 128)";
        case W4_ERR_MISALIGNED: return "W4_ERR_MISALIGNED: pointer alignment violated";
        case W4_ERR_CUDA: return "W4_ERR_CUDA: CUDA call or kernel launch failed";
        case W4_ERR_TIMEOUT: return "W4_ERR_TIMEOUT: a kernel gave up a bounded wait";
        case W4_ERR_SCRATCH_LIMIT:
            return "W4_ERR_SCRATCH_LIMIT: the call needs more scratch than the library's fixed array holds";
        default: return "unknown w4a16 status";
    }
}

int w4_quantize_pack(const void *W, int w_dtype, int64_t N, int64_t K, int group,
                     uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream) {
    return quantize_pack_impl<false>(W, w_dtype, N, K, group, qweight, scales, zeros, stream);
}

int w4_quantize_pack_sym(const void *W, int w_dtype, int64_t N, int64_t K, int group,
                         uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream) {
    return quantize_pack_impl<true>(W, w_dtype, N, K, group, qweight, scales, zeros, stream);
}

int w4_quantize_pack_percentile(const void *W, int w_dtype, int64_t N, int64_t K, int group, float p,
                                uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream) {
    return quantize_calib_impl(false, W, w_dtype, N, K, group, p, 0, qweight, scales, zeros, stream);
}

int w4_quantize_pack_mse(const void *W, int w_dtype, int64_t N, int64_t K, int group, int candidates,
                         uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream) {
    return quantize_calib_impl(true, W, w_dtype, N, K, group, 0.0f, candidates, qweight, scales, zeros, stream);
}

int w4_dequantize(const uint8_t *qweight, const void *scales, const uint8_t *zeros, int64_t N, int64_t K,
                  int group, int out_dtype, void *out, cudaStream_t stream) {
    if (N < 0 || K < 0 || group <= 0) return W4_ERR_INVALID_ARG;
    if (out_dtype != W4_DTYPE_BF16 && out_dtype != W4_DTYPE_F16) return W4_ERR_INVALID_ARG;
    if (group != W4_GROUP_SIZE) return W4_ERR_UNSUPPORTED;
    if (K % group != 0) return W4_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return W4_OK;
    if (!qweight || !scales || !zeros || !out) return W4_ERR_INVALID_ARG;
    if (!aligned(qweight, 16) || !aligned(scales, 2) || !aligned(out, 16)) return W4_ERR_MISALIGNED;
    if (N > INT64_MAX / K) return W4_ERR_INVALID_ARG;
    int sms = 0;
    if (int rc = current_sm_count(&sms)) return rc;
    namespace dq = w4::deq;
    const int64_t chunks = N * K / 8;                  // 8 levels per chunk
    const int64_t per_block = static_cast<int64_t>(dq::NUM_THREADS) * dq::UNROLL;
    int64_t blocks = (chunks + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(sms) * dq::BLOCKS_PER_SM;
    if (blocks > cap) blocks = cap;
    const uint32_t *qw = reinterpret_cast<const uint32_t *>(qweight);
    const __half *sc = static_cast<const __half *>(scales);
    uint4 *o = static_cast<uint4 *>(out);
    if (out_dtype == W4_DTYPE_BF16)
        return launch(dq::dequantize_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(dq::NUM_THREADS), 0,
                      stream, qw, sc, zeros, o, chunks);
    return launch(dq::dequantize_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(dq::NUM_THREADS), 0,
                  stream, qw, sc, zeros, o, chunks);
}

int w4_matmul(const void *A, int64_t M, int64_t N, int64_t K, int group, const uint8_t *qweight,
              const void *scales, const uint8_t *zeros, void *Y, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0 || group <= 0) return W4_ERR_INVALID_ARG;
    if (group != W4_GROUP_SIZE) return W4_ERR_UNSUPPORTED;
    if (K % group != 0) return W4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4_OK;
    if (!Y) return W4_ERR_INVALID_ARG;
    if (!aligned(Y, 2)) return W4_ERR_MISALIGNED;
    if (K == 0) {
        const cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(M * N) * 2, stream);
        return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
    }
    if (!A || !qweight || !scales || !zeros) return W4_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(qweight, 16) || !aligned(scales, 2)) return W4_ERR_MISALIGNED;
    int sms = 0;
    if (int rc = current_sm_count(&sms)) return rc;
    const __nv_bfloat16 *a = static_cast<const __nv_bfloat16 *>(A);
    const __half *s = static_cast<const __half *>(scales);
    __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(Y);
    // Decode shapes (2 <= M <= 16): warp-level MMAs on weights dequantized in registers,
    // whenever K is a multiple of 2048 and the activations fit in shared memory.  (M = 1
    // stays on the integer-dot GEMV, faster there: 7.1 against 9.0 us on 11008 x 4096.)
    if (M >= 2 && M <= 16) {
        const int rc = launch_gemv_mma(a, false, nullptr, M, N, K, qweight, s, zeros, y, stream, sms, wait_params(),
                                       false);
        if (rc != W4_ERR_UNSUPPORTED) return rc;
    }
    if (M <= 8) return launch_gemv(a, M, N, K, qweight, s, zeros, y, stream, sms, wait_params());
    return w4::launch_gemm_tcgen05(a, M, N, K, qweight, s, zeros, y, stream, sms, wait_params());
}

int w4_quantize_act_int8(const void *A, int64_t M, int64_t K, int8_t *a_q, float *a_scale, cudaStream_t stream) {
    if (M < 0 || K < 0 || K % 8 != 0) return W4_ERR_INVALID_ARG;
    if (M == 0) return W4_OK;
    if (!a_scale || (K > 0 && (!A || !a_q))) return W4_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(a_q, 16) || !aligned(a_scale, 4)) return W4_ERR_MISALIGNED;
    if (M > INT64_MAX / (K > 0 ? K : 1)) return W4_ERR_INVALID_ARG;
    int sms = 0;
    if (int rc = current_sm_count(&sms)) return rc;
    namespace aq = w4::actq;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (M <= 2 * static_cast<int64_t>(sms))       // few rows: 256 threads on each
        return launch(aq::act_quant_int8_kernel, dim3(static_cast<unsigned>(M)), dim3(aq::NUM_THREADS), 0, stream,
                      static_cast<const __nv_bfloat16 *>(A), M, K, a_q, a_scale);
    int64_t blocks = (M + 7) / 8;                  // many rows: a warp on each
    if (blocks > cap) blocks = cap;
    return launch(aq::act_quant_int8_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(aq::NUM_THREADS), 0,
                  stream, static_cast<const __nv_bfloat16 *>(A), M, K, a_q, a_scale);
}

size_t w4_matmul_w4a8_workspace_size(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0 || gemv_mma_shape_ok(M, K)) return 0;
    if (M > INT64_MAX / 2 / K) return 0;
    return static_cast<size_t>((M * K * 2 + 255) / 256 * 256);
}

int w4_matmul_w4a8(const int8_t *a_q, const float *a_scale, int64_t M, int64_t N, int64_t K, int group,
                   const uint8_t *qweight, const void *scales, const uint8_t *zeros, void *Y, void *workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0 || group <= 0) return W4_ERR_INVALID_ARG;
    if (group != W4_GROUP_SIZE) return W4_ERR_UNSUPPORTED;
    if (K % group != 0) return W4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4_OK;
    if (!Y) return W4_ERR_INVALID_ARG;
    if (!aligned(Y, 2)) return W4_ERR_MISALIGNED;
    if (K == 0) {
        const cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(M * N) * 2, stream);
        return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
    }
    if (!a_q || !a_scale || !qweight || !scales || !zeros) return W4_ERR_INVALID_ARG;
    if (!aligned(a_q, 16) || !aligned(a_scale, 4) || !aligned(qweight, 16) || !aligned(scales, 2))
        return W4_ERR_MISALIGNED;
    int sms = 0;
    if (int rc = current_sm_count(&sms)) return rc;
    const __half *s = static_cast<const __half *>(scales);
    __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(Y);
    if (M == 1) {                  // one token: integer dot products on the int8 digits
        const int rc = launch_gemv_dp4a(a_q, true, a_scale, N, K, qweight, s, zeros, y, stream, sms, wait_params());
        if (rc != W4_ERR_UNSUPPORTED) return rc;
    }
    if (gemv_mma_shape_ok(M, K))   // decode shapes: widened while staged, no workspace
        return launch_gemv_mma(a_q, true, a_scale, M, N, K, qweight, s, zeros, y, stream, sms, wait_params(), true);
    // Other shapes: a_q widened (exactly) to bf16 in the workspace, then the tcgen05 GEMM
    // with the per-row activation scale applied in its epilogue.
    const size_t need = w4_matmul_w4a8_workspace_size(M, K);
    if (!workspace || workspace_bytes < need) return W4_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return W4_ERR_MISALIGNED;
    __nv_bfloat16 *abf = static_cast<__nv_bfloat16 *>(workspace);
    const int64_t n8 = M * K / 8;
    int64_t blocks = (n8 + 255) / 256;
    if (blocks > static_cast<int64_t>(sms) * 16) blocks = static_cast<int64_t>(sms) * 16;
    if (int rc = launch(w4::actq::int8_to_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, a_q,
                        abf, n8))
        return rc;
    return w4::launch_gemm_tcgen05(abf, M, N, K, qweight, s, zeros, y, stream, sms, wait_params(), a_scale);
}

int w4_matmul_w4a8_noalloc(const int8_t *a_q, const float *a_scale, int64_t M, int64_t N, int64_t K, int group,
                           const uint8_t *qweight, const void *scales, const uint8_t *zeros, void *Y,
                           cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0 || group <= 0) return W4_ERR_INVALID_ARG;
    if (group != W4_GROUP_SIZE) return W4_ERR_UNSUPPORTED;
    if (K % group != 0) return W4_ERR_INVALID_ARG;
    const size_t need = w4_matmul_w4a8_workspace_size(M, K);
    if (need > W4_NOALLOC_SCRATCH_BYTES) return W4_ERR_SCRATCH_LIMIT;   // before anything is launched
    void *scratch = nullptr;
    if (need > 0 && M > 0 && N > 0) {
        if (int rc = noalloc_scratch(&scratch)) return rc;
    }
    return w4_matmul_w4a8(a_q, a_scale, M, N, K, group, qweight, scales, zeros, Y, scratch, need, stream);
}

int w4_gptq_quantize(const void *W, int w_dtype, int64_t N, int64_t K, int group, const float *U,
                     uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream) {
    if (N < 0 || K < 0 || group <= 0) return W4_ERR_INVALID_ARG;
    if (w_dtype != W4_DTYPE_F16 && w_dtype != W4_DTYPE_F32) return W4_ERR_INVALID_ARG;
    if (group != W4_GROUP_SIZE) return W4_ERR_UNSUPPORTED;
    if (K % group != 0) return W4_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return W4_OK;
    if (K > 8192 || N > INT32_MAX / 2) return W4_ERR_UNSUPPORTED;
    if (!W || !U || !qweight || !scales || !zeros) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(U, 16) || !aligned(qweight, 16) || !aligned(scales, 2))
        return W4_ERR_MISALIGNED;
    namespace gq = w4::gptq;
    gq::Params prm;
    prm.W = W;
    prm.U = U;
    prm.qweight = qweight;
    prm.scales = static_cast<__half *>(scales);
    prm.zeros = zeros;
    prm.N = static_cast<int>(N);
    prm.K = static_cast<int>(K);
    prm.R = gq::rows_for(prm.K);
    const int smem = gq::smem_bytes(prm.K, prm.R);
    const int64_t grid = (N + prm.R - 1) / prm.R;
    auto kern = w_dtype == W4_DTYPE_F32 ? gq::gptq_kernel<true> : gq::gptq_kernel<false>;
    if (int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem)) return rc;
    return launch(kern, dim3(static_cast<unsigned>(grid)), dim3(gq::NUM_THREADS), smem, stream, prm);
}

int w4_check_device_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return W4_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, w4::g_error_word, sizeof(word)) != cudaSuccess) return W4_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(w4::g_error_word, &zero, sizeof(zero)) != cudaSuccess) return W4_ERR_CUDA;
        return static_cast<int>(word);
    }
    return W4_OK;
}

void w4_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns ? ns : 2000000000ull, std::memory_order_relaxed);
}

void w4_debug_inject_stall(int enable) { g_stall.store(enable ? 1 : 0, std::memory_order_relaxed); }

}  // extern "C"
