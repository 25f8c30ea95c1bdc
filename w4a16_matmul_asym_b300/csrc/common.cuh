// common.cuh -- device helpers shared by the kernels of libw4a16 (sm_103a only).
//
// Everything that waits is bounded: a wait that does not complete within the
// caller-given number of nanoseconds of %globaltimer records W4_ERR_TIMEOUT in the
// device error word, raises the CTA's abort flag and returns false, so kernels can
// drain their in-flight copies, free tensor memory and exit without trapping.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "w4a16.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libw4a16 targets sm_103a only"
#endif

namespace w4 {

// One error word per device for the whole library (read by w4_check_device_error).
__device__ unsigned int g_error_word;

// Launch-time knobs shared by every kernel.
struct WaitParams {
    unsigned long long timeout_ns;  // limit of each bounded wait
    int stall;                      // test hook: wait on a barrier nobody signals
};

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(unsigned int code) {
    atomicCAS(&g_error_word, 0u, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed.  Returns false
// if the CTA's abort flag is raised or the wait runs out of time (which raises the
// flag and records W4_ERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned long long timeout_ns) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                record_error(W4_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait for roles off the critical path (producer refills, epilogue): between
// polls the thread backs off with __nanosleep (16 ns doubling to 256 ns), so it takes
// few issue slots from the consumer warps sharing its SM sub-partition.
__device__ __forceinline__ bool mbar_wait_polite(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                 unsigned long long timeout_ns) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    unsigned int ns = 16;
    for (;;) {
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
        if (mbar_try_wait(a, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            record_error(W4_ERR_TIMEOUT);
            return false;
        }
    }
}

// ---- bulk / tensor copies (TMA) ---------------------------------------------------
// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 2-D tiled tensor copy global -> shared.  x is the innermost coordinate; x times the
// element size must be a multiple of 16 bytes (callers only pass such x).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// reads (tensor-core operand fetches) of the same addresses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tensor store shared -> global (async proxy), tracked in this thread's bulk group.
// The box is clipped at the tensor's edges; x and y must be >= 0 and x * element size a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int32_t x,
                                             int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_addr(src)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's committed bulk stores have finished reading their shared-memory source.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_group0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- programmatic dependent launch --------------------------------------------------
// Kernels launched with programmatic stream serialization call this before touching
// global memory: it waits until the preceding kernel in the stream has completed and
// its writes are visible, then lets the next kernel begin launching (it will wait the
// same way).  Without that launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- misc ---------------------------------------------------------------------
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// Bounded wait of a whole, converged warp.  Every lane polls the barrier and a vote
// decides, so the warp never splits into a polling lane and 31 lanes parked on a
// shuffle: that pattern (one lane waits, then __shfl_sync broadcasts the outcome)
// measured 20-40 % slower in the tensor-core kernels, whose producer, MMA and
// dequantize warps wait once or more per k-block.  On a timeout (or a raised abort
// flag) lane 0 records W4_ERR_TIMEOUT and every lane returns false; with `polite` the
// lanes back off with __nanosleep between polls (16 ns doubling to 256 ns).
__device__ __forceinline__ bool warp_mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                               unsigned long long timeout_ns, bool polite = false) {
    const uint32_t a = smem_addr(bar);
    if (__all_sync(0xffffffffu, mbar_try_wait(a, parity))) return true;
    const unsigned long long t0 = globaltimer_ns();
    unsigned int ns = 16;
    for (uint32_t it = 1;; ++it) {
        if (polite) {
            __nanosleep(ns);
            if (ns < 256) ns <<= 1;
        }
        if (__all_sync(0xffffffffu, mbar_try_wait(a, parity))) return true;
        if (polite || (it & 15u) == 0) {
            int stop = 0;
            if (lane_id() == 0) {
                if (*abort_flag) {
                    stop = 1;
                } else if (globaltimer_ns() - t0 > timeout_ns) {
                    *abort_flag = 1;
                    record_error(W4_ERR_TIMEOUT);
                    stop = 1;
                }
            }
            if (__any_sync(0xffffffffu, stop)) return false;
        }
    }
}

__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Streaming 16-byte global load that does not allocate in L1 (read-once data).
__device__ __forceinline__ uint4 ldg_stream_16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace w4
