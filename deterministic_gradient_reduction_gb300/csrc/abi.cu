// C-ABI glue: status strings, version, device check, device status word.
#include "dgr_common.cuh"

namespace dgr {

dgr_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGR_ERR_CUDA;
    return dgr_device_supported(dev);
}

}  // namespace dgr

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
