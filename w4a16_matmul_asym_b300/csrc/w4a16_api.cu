// w4a16_api.cu -- the extern "C" entry points of libw4a16 (see include/w4a16.h).
//
// One translation unit holds every kernel, so the device error word is a single
// symbol.  The entry points validate arguments on the host, pick a kernel, and
// enqueue it on the caller's stream with cudaLaunchKernelEx (whose return value is
// the launch status); they never synchronize and never allocate.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "gemm_tcgen05.cuh"
#include "gemv.cuh"
#include "quantize_pack.cuh"

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

int launch_gemv(const __nv_bfloat16 *A, int64_t M, int64_t N, int64_t K, const uint8_t *qweight,
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
        default: return "unknown w4a16 status";
    }
}

int w4_quantize_pack(const void *W, int w_dtype, int64_t N, int64_t K, int group,
                     uint8_t *qweight, void *scales, uint8_t *zeros, cudaStream_t stream) {
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
    // 8 groups per warp iteration, 8 warps per block; at most 8 resident blocks per SM.
    int64_t blocks = (total_groups + 63) / 64;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    uint32_t *qw = reinterpret_cast<uint32_t *>(qweight);
    __half *sc = static_cast<__half *>(scales);
    if (w_dtype == W4_DTYPE_F16)
        return launch(w4::quantize_pack_kernel<false>, grid, block, 0, stream, W, total_groups, qw, sc, zeros);
    return launch(w4::quantize_pack_kernel<true>, grid, block, 0, stream, W, total_groups, qw, sc, zeros);
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
    if (M <= 8) return launch_gemv(a, M, N, K, qweight, s, zeros, y, stream, sms);
    return w4::launch_gemm_tcgen05(a, M, N, K, qweight, s, zeros, y, stream, sms, wait_params());
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
