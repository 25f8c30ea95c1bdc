// prefetch.cuh -- L2 prefetch of read-only kernel inputs, issued ahead of the
// dependency wait of programmatic dependent launch (sm_103a only).
#pragma once

#include "common.cuh"

namespace w4 {

// ---- L2 prefetch ahead of the dependency wait ------------------------------------
// Asks L2 to start fetching bytes [begin, end) of a buffer (offsets rounded down to 16
// bytes, so the range never leaves the buffer; skipped unless the base is 16-byte
// aligned).  A prefetch writes nothing and hands nothing to the CTA, so a kernel may issue
// it before pdl_wait_then_release(): the hardware keeps L2 coherent, and the loads made
// after the wait still see every write of the preceding kernel.  Kernels prefetch only
// their read-only weight inputs this way, while the preceding kernel drains.
__device__ __forceinline__ void prefetch_l2_range(const void *base, int64_t begin, int64_t end) {
    const uint64_t b = reinterpret_cast<uint64_t>(base);
    if (b & 15u) return;
    begin &= ~static_cast<int64_t>(15);
    end &= ~static_cast<int64_t>(15);
    for (int64_t off = begin; off < end; off += 32768) {
        const uint32_t sz = static_cast<uint32_t>(end - off < 32768 ? end - off : 32768);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(b + off), "r"(sz) : "memory");
    }
}
// The first `cap` bytes of the packed rows [r0, r1) of a [N, K/2] weight matrix, and
// the scale / zero-point rows they cover.
__device__ __forceinline__ void prefetch_weight_band_l2(const uint8_t *qweight, const __half *scales,
                                                        const uint8_t *zeros, int64_t r0, int64_t r1, int64_t K,
                                                        int64_t cap) {
    if (r1 <= r0 || K <= 0) return;
    const int64_t rowq = K / 2, ngr = K / 128;
    const int64_t nq = (r1 - r0) * rowq < cap ? (r1 - r0) * rowq : cap;
    prefetch_l2_range(qweight, r0 * rowq, r0 * rowq + nq);
    const int64_t rows = (nq + rowq - 1) / rowq;
    prefetch_l2_range(scales, r0 * ngr * 2, (r0 + rows) * ngr * 2);
    prefetch_l2_range(zeros, r0 * ngr, (r0 + rows) * ngr);
}

}  // namespace w4
