// C-ABI glue: status strings, version, device check, device status word, the
// diagnostic launch schedule and the usable SM count.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "dgr_common.cuh"
#include "dgr_diag.h"

namespace dgr {

dgr_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGR_ERR_CUDA;
    return dgr_device_supported(dev);
}

namespace {

std::atomic<int32_t> g_order{0};
std::atomic<int32_t> g_cap{0};
std::atomic<uint32_t> g_seed{0};

// cuCtxGetCurrent and cuCtxGetDevResource through the runtime's driver entry
// points (no link to libcuda); null when the driver does not offer them.
using CtxGetCurrent = CUresult (*)(CUcontext *);
using CtxGetDevResource = CUresult (*)(CUcontext, CUdevResource *, CUdevResourceType);
CtxGetCurrent g_get_cur = nullptr;
CtxGetDevResource g_get_res = nullptr;
std::once_flag g_driver_once;

void *driver_entry(const char *name, int version) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return f;
}

}  // namespace

Sched sched_setting() {
    Sched s{};
    s.order = g_order.load(std::memory_order_relaxed);
    s.cap = g_cap.load(std::memory_order_relaxed);
    s.seed = g_seed.load(std::memory_order_relaxed);
    s.n = 0;
    s.a = 1;
    s.b = 0;
    return s;
}

Sched sched_for(uint32_t n) { return sched_over(sched_setting(), n); }

unsigned sched_grid(unsigned grid) {
    const int32_t cap = g_cap.load(std::memory_order_relaxed);
    return (cap > 0 && static_cast<unsigned>(cap) < grid) ? static_cast<unsigned>(cap) : grid;
}

dgr_status usable_sms(int *sms) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DGR_ERR_CUDA;
    std::call_once(g_driver_once, [] {
        g_get_cur = reinterpret_cast<CtxGetCurrent>(driver_entry("cuCtxGetCurrent", 12000));
        g_get_res = reinterpret_cast<CtxGetDevResource>(driver_entry("cuCtxGetDevResource", 12040));
    });
    CUcontext ctx = nullptr;
    CUdevResource r{};
    // a green context's SM partition, when the current context is one
    if (g_get_cur && g_get_res && g_get_cur(&ctx) == CUDA_SUCCESS && ctx &&
        g_get_res(ctx, &r, CU_DEV_RESOURCE_TYPE_SM) == CUDA_SUCCESS && r.sm.smCount > 0 &&
        static_cast<int>(r.sm.smCount) < n)
        n = static_cast<int>(r.sm.smCount);
    const int32_t cap = g_cap.load(std::memory_order_relaxed);
    if (cap > 0 && cap < n) n = cap;
    *sms = n;
    return DGR_OK;
}

}  // namespace dgr

extern "C" dgr_status dgr_diag_set_schedule(int32_t order, uint32_t seed, int32_t grid_cap) {
    if (order < 0 || order > 2 || grid_cap < 0) return DGR_ERR_INVALID_ARG;
    dgr::g_order.store(order);
    dgr::g_seed.store(seed);
    dgr::g_cap.store(grid_cap);
    return DGR_OK;
}

extern "C" const char *dgr_status_string(dgr_status s) {
    switch (s) {
        case DGR_OK: return "DGR_OK";
        case DGR_ERR_INVALID_ARG: return "DGR_ERR_INVALID_ARG";
        case DGR_ERR_UNSUPPORTED: return "DGR_ERR_UNSUPPORTED";
        case DGR_ERR_WORKSPACE_TOO_SMALL: return "DGR_ERR_WORKSPACE_TOO_SMALL";
        case DGR_ERR_ALIAS: return "DGR_ERR_ALIAS";
        case DGR_ERR_MISALIGNED: return "DGR_ERR_MISALIGNED";
        case DGR_ERR_CUDA: return "DGR_ERR_CUDA";
        case DGR_ERR_TIMEOUT: return "DGR_ERR_TIMEOUT";
        default: return "DGR_ERR_UNKNOWN";
    }
}

extern "C" int32_t dgr_version(void) { return 103; }

extern "C" dgr_status dgr_device_supported(int32_t device) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) {
        cudaGetLastError();
        return DGR_ERR_UNSUPPORTED;
    }
    return (major == 10 && minor == 3) ? DGR_OK : DGR_ERR_UNSUPPORTED;
}

extern "C" dgr_status dgr_read_device_status(const void *ws, int32_t clear, int32_t *status, void *stream) {
    if (!ws || !status) return DGR_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return DGR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DGR_ERR_CUDA;
    *status = v;
    if (clear && v != 0) {
        if (cudaMemsetAsync(const_cast<void *>(ws), 0, sizeof(dgr::WsHeader), s) != cudaSuccess)
            return DGR_ERR_CUDA;
    }
    return DGR_OK;
}

extern "C" dgr_status dgr_query_device_status(const void *ws, void *stream) {
    int32_t v = 0;
    const dgr_status r = dgr_read_device_status(ws, 0, &v, stream);
    return r != DGR_OK ? r : static_cast<dgr_status>(v);
}
