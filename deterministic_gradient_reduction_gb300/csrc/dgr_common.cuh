// Shared device/host helpers for the dgr kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dgr.h"

namespace dgr {

// Every workspace starts with this header; the rest is per-operation.
struct WsHeader {
    int32_t status;     // first device-side error code (0 = none)
    int32_t where;      // diagnostic: which wait gave up
    int32_t pad[62];    // per-operation tickets and accumulators
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000ull * 1000ull * 1000ull;  // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t *p) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void record_error(WsHeader *h, int32_t code, int32_t where) {
    if (atomicCAS(&h->status, 0, code) == 0) atomicExch(&h->where, where);
}

// Spin until *p >= target (acquire), at most kWaitLimitNs. Returns false on timeout.
__device__ __forceinline__ bool wait_counter_geq(const int32_t *p, int32_t target) {
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    unsigned ns = 32;
    while (true) {
        __nanosleep(ns);
        if (ld_acquire_gpu(p) >= target) return true;
        if (ns < 1024) ns <<= 1;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// 16-byte read-only load of data that no kernel writes during the launch.
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Host side -------------------------------------------------------------------

inline bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

inline bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks the current device is compute capability 10.3.
dgr_status check_device();

inline dgr_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DGR_OK : DGR_ERR_CUDA;
}

}  // namespace dgr
