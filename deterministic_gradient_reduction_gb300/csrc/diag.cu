// A bounded wait that runs out on purpose (see dgr_diag.h): the failure
// path of the library's waits, exercised without a fault or a hang.
#include "tc_common.cuh"
#include "dgr_diag.h"

namespace dgr {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int which, uint64_t limit_ns, WsHeader *hdr) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    if (which == 0) {
        // pad[1] of a zeroed workspace: nothing ever increments it
        if (!wait_counter_geq(&hdr->pad[1], 1, limit_ns)) record_error(hdr, DGR_ERR_TIMEOUT, 90);
    } else {
        abort_flag = 0;
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
        // nobody arrives: phase 0 never completes
        tc::mbar_wait(&bar, 0, &abort_flag, hdr, 91, limit_ns);
    }
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" dgr_status dgr_diag_wait_timeout(int32_t which, int32_t limit_us, void *ws, size_t ws_bytes,
                                            void *stream) {
    if ((which != 0 && which != 1) || limit_us < 1 || limit_us > 1000000 || !ws) return DGR_ERR_INVALID_ARG;
    if (ws_bytes < sizeof(WsHeader)) return DGR_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(ws, kAlign)) return DGR_ERR_MISALIGNED;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        which, static_cast<uint64_t>(limit_us) * 1000ull, static_cast<WsHeader *>(ws));
    return launch_status();
}

extern "C" dgr_status dgr_diag_noalloc_wait_timeout(int32_t which, int32_t limit_us, void *stream) {
    if ((which != 0 && which != 1) || limit_us < 1 || limit_us > 1000000) return DGR_ERR_INVALID_ARG;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    void *ws = nullptr;
    if ((st = noalloc_scratch(&ws)) != DGR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), s) != cudaSuccess) return DGR_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, s>>>(which, static_cast<uint64_t>(limit_us) * 1000ull,
                                         static_cast<WsHeader *>(ws));
    return launch_status();
}
