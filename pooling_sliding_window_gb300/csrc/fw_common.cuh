// fw_common.cuh -- internal helpers shared by the libfusedwin translation units.
// Not part of the public ABI (include/fusedwin.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fusedwin.h"

namespace fw {

// Device-side error bits, OR-ed into a per-translation-unit error word.
enum : unsigned {
    DEVERR_TIMEOUT = 1u,   // a bounded mbarrier wait gave up
    DEVERR_INTERNAL = 2u,  // an internal consistency check failed
};

// Devices for which per-device state is cached.
constexpr int FW_MAX_DEVICES = 64;

// Wall-clock limit of a bounded wait inside a kernel.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s

// Launch bookkeeping (host side, fw_api.cu).
void note_launch(int n = 1);
fw_status launch_status(cudaError_t e);

// ---------------------------------------------------------------- device --

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Running max of the MaxPool2d definition: a larger value or a NaN replaces the
// current value unless that is already NaN; ties keep the current (earlier) tap.
__device__ __forceinline__ float max_update(float m, float v) {
    return (m == m && !(v <= m)) ? v : m;
}
// Mirror rule for a running minimum (used when the scale is negative).
__device__ __forceinline__ float min_update(float m, float v) {
    return (m == m && !(v >= m)) ? v : m;
}

// ------------------------------------------------------------- mbarriers --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after WAIT_LIMIT_NS.
// Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
}

// 1-D bulk copy global -> shared (TMA engine), completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

}  // namespace fw
