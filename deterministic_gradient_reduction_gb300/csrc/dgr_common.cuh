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

// Spin until *p >= target (acquire), at most limit_ns. Returns false on timeout.
__device__ __forceinline__ bool wait_counter_geq(const int32_t *p, int32_t target, uint64_t limit_ns = kWaitLimitNs) {
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    unsigned ns = 32;
    while (true) {
        __nanosleep(ns);
        if (ld_acquire_gpu(p) >= target) return true;
        if (ns < 1024) ns <<= 1;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Which CTA (or warp) takes which work item. The product path hands items out
// in ascending order over as many CTAs as it needs; a test can ask, through
// dgr_diag_set_schedule(), for descending or shuffled order and for a capped
// grid, to show that no result depends on it. Item i of n is then
//   ascending: i;  descending: n - 1 - i;  shuffled: (a * i + b) mod n,
// with a coprime to n (a bijection of [0, n)).
struct Sched {
    int32_t order;  // 0 ascending, 1 descending, 2 shuffled
    int32_t cap;    // > 0: launches take at most this many CTAs
    uint32_t seed;
    uint32_t n, a, b;
};

// The schedule over n items (a and b from the seed; the order falls back to
// ascending for n <= 1). On the device for item counts only the GPU knows.
__host__ __device__ inline Sched sched_over(Sched s, uint32_t n) {
    s.n = n;
    s.a = 1;
    s.b = 0;
    if (n <= 1) s.order = 0;
    if (s.order == 2) {
        uint32_t a = ((s.seed * 2654435761u) | 1u) % n;
        if (a == 0) a = 1;
        for (;;) {  // the next multiplier coprime to n (1 always is)
            uint32_t x = a, y = n;
            while (y) {
                const uint32_t t = x % y;
                x = y;
                y = t;
            }
            if (x == 1) break;
            a = a + 1 < n ? a + 1 : 1;
        }
        s.a = a;
        s.b = (s.seed ^ 0x9e3779b9u) % n;
    }
    return s;
}

__device__ __forceinline__ uint32_t sched_item(const Sched &s, uint32_t i) {
    if (s.order == 0) return i;
    if (s.order == 1) return s.n - 1u - i;
    return static_cast<uint32_t>((static_cast<uint64_t>(s.a) * i + s.b) % s.n);
}

// Two binary32 adds in one packed instruction (add.rn.f32x2): each half is
// rounded to nearest even with subnormals kept, so d.x, d.y carry the same
// bits as __fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y) (checked on the GPU over 4
// million operand pairs, a quarter of them subnormal); half the issue slots.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Two binary32 products in one packed instruction (mul.rn.f32x2), likewise
// the same bits as two __fmul_rn (checked over 4 million operand pairs, an
// eighth of the products subnormal). A packed product may feed scalar
// __fadd_rn adds (both roundings kept, checked likewise) but never a packed
// add: the code generator fuses mul.rn.f32x2 followed by add.rn.f32x2 into a
// fused multiply-add (a quarter of 2 million normal-operand results came out
// with the fused rounding), so add2(c, mul2(a, b)) is not written anywhere.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// d[e] = a[e] + b[e] (binary32, round to nearest even) for e < n, in pairs.
template <int n>
__device__ __forceinline__ void vadd(float *d, const float *a, const float *b) {
#pragma unroll
    for (int e = 0; e + 1 < n; e += 2) {
        const float2 r = add2(make_float2(a[e], a[e + 1]), make_float2(b[e], b[e + 1]));
        d[e] = r.x;
        d[e + 1] = r.y;
    }
    if (n & 1) d[n - 1] = __fadd_rn(a[n - 1], b[n - 1]);
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

// Predicated loads: the destination keeps its value when pred is false. The
// predicate lives inside the asm with the destination as an in-out operand,
// so nothing has to merge the old and the new value (a merge would wait for
// the load to land and serialise loads meant to be in flight together).
__device__ __forceinline__ void ldg_nc_v4f_if(float4 &v, const void *ptr, bool pred) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];\n\t}"
        : "+f"(v.x), "+f"(v.y), "+f"(v.z), "+f"(v.w)
        : "l"(ptr), "r"(static_cast<int>(pred)));
}

// Same, L2 only (.cg): data written earlier in this launch by other blocks.
__device__ __forceinline__ void ldcg_v4f_if(float4 &v, const void *ptr, bool pred) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];\n\t}"
        : "+f"(v.x), "+f"(v.y), "+f"(v.z), "+f"(v.w)
        : "l"(ptr), "r"(static_cast<int>(pred)));
}

// Same, plain weak load (data this thread may also write).
__device__ __forceinline__ void ld_v4f_if(float4 &v, const void *ptr, bool pred) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q ld.global.v4.f32 {%0,%1,%2,%3}, [%4];\n\t}"
        : "+f"(v.x), "+f"(v.y), "+f"(v.z), "+f"(v.w)
        : "l"(ptr), "r"(static_cast<int>(pred)));
}

// 16-byte read-only integer load under a predicate.
__device__ __forceinline__ void ldg_nc_v4u_if(uint4 &v, const void *ptr, bool pred) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
        : "l"(ptr), "r"(static_cast<int>(pred)));
}

// 32-bit read-only load under a predicate.
__device__ __forceinline__ void ldg_nc_b32_if(int32_t &v, const int32_t *ptr, bool pred) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q ld.global.nc.b32 %0, [%1];\n\t}"
        : "+r"(v)
        : "l"(ptr), "r"(static_cast<int>(pred)));
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

// The process-wide diagnostic setting (ascending and uncapped unless a test
// changed it), not yet bound to an item count.
Sched sched_setting();

// The schedule for a launch over n work items: sched_over(sched_setting(), n).
Sched sched_for(uint32_t n);

// grid, capped by the diagnostic setting.
unsigned sched_grid(unsigned grid);

// SMs that the kernels of the current context can hold at once: the device's,
// or the SM partition of a green context, lowered to the diagnostic grid cap.
// Persistent kernels whose CTAs wait on one another size their grids by it.
dgr_status usable_sms(int *sms);

// Device address, on the current device, of the column sum's static scratch
// array (the no-alloc entry's scratch); looked up once per device.
dgr_status noalloc_scratch(void **ptr);

inline dgr_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DGR_OK : DGR_ERR_CUDA;
}

}  // namespace dgr
