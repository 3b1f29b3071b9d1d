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

// Controls for the replay tests: the order-varying reductions the pages
// replace. Each CTA sums its own part in a fixed order and then adds it to
// the output with a float atomicAdd, so the order in which the parts arrive,
// and with it the rounding, follows the scheduling of the CTAs.
constexpr int kAtomicRows = 128;

// Column sum, x bf16 [T, H] row-major: one CTA per tile of 128 rows, thread h
// of the CTA sums column h of its rows in order, then one atomicAdd per column.
__global__ void __launch_bounds__(256) atomic_colsum_kernel(const uint16_t *x, int64_t T, int32_t H, float *out) {
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kAtomicRows;
    const int64_t t1 = min(t0 + kAtomicRows, T);
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        float acc = 0.0f;
        for (int64_t t = t0; t < t1; ++t) acc = __fadd_rn(acc, bf16_bits_to_f32(x[t * H + h]));
        atomicAdd(out + h, acc);
    }
}

// dprob, dY and Y bf16 [M, N] row-major: CTA (N-tile of 128, row block): a
// warp per row sums its tile's products, lane by lane then by shuffles, and
// adds the tile's partial to dprob[m] with one atomicAdd. The N-tile is the
// fastest grid index, so a row's tiles run side by side on different SMs and
// their atomics race (with the row block fastest, a row's tiles would run in
// launch order, one wave after another, and the sum would look stable).
__global__ void __launch_bounds__(256) atomic_rowdot_kernel(const uint16_t *dY, const uint16_t *Y, int64_t M,
                                                           int32_t N, float *dprob) {
    const int lane = threadIdx.x & 31;
    const int64_t m = static_cast<int64_t>(blockIdx.y) * 8 + (threadIdx.x >> 5);
    if (m >= M) return;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
    float v = 0.0f;
    for (int64_t c = c0 + lane; c < min(c0 + 128, static_cast<int64_t>(N)); c += 32)
        v = __fadd_rn(v, __fmul_rn(bf16_bits_to_f32(dY[m * N + c]), bf16_bits_to_f32(Y[m * N + c])));
    for (int d = 16; d; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
    if (lane == 0) atomicAdd(dprob + m, v);
}

// Packed binary32 arithmetic as the kernels use it: add2 / mul2 on pairs.
__global__ void __launch_bounds__(256) packed_ops_kernel(const float2 *a, const float2 *b, int64_t n, float2 *sum,
                                                         float2 *prod) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        sum[i] = add2(a[i], b[i]);
        prod[i] = mul2(a[i], b[i]);
    }
}

// A packed product feeding binary32 round-to-nearest adds, as the dsReLU
// leaves feed their tree: chain = c + RN(a * b), two values at a time.
__global__ void __launch_bounds__(256) packed_chain_kernel(const float2 *a, const float2 *b, const float2 *c, int64_t n,
                                                           float2 *chain) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float2 pr = mul2(a[i], b[i]);
        chain[i] = make_float2(__fadd_rn(c[i].x, pr.x), __fadd_rn(c[i].y, pr.y));
    }
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" dgr_status dgr_diag_packed_chain(const float *a, const float *b, const float *c, int64_t n_pairs,
                                            float *chain, void *stream) {
    if (n_pairs < 0 || (n_pairs > 0 && (!a || !b || !c || !chain))) return DGR_ERR_INVALID_ARG;
    if (!aligned(a, 8) || !aligned(b, 8) || !aligned(c, 8) || !aligned(chain, 8)) return DGR_ERR_MISALIGNED;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    if (n_pairs == 0) return DGR_OK;
    const int64_t blocks = (n_pairs + 255) / 256;
    packed_chain_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0,
                          static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float2 *>(a), reinterpret_cast<const float2 *>(b), reinterpret_cast<const float2 *>(c),
        n_pairs, reinterpret_cast<float2 *>(chain));
    return launch_status();
}

extern "C" dgr_status dgr_diag_packed_ops(const float *a, const float *b, int64_t n_pairs, float *sum, float *prod,
                                          void *stream) {
    if (n_pairs < 0 || (n_pairs > 0 && (!a || !b || !sum || !prod))) return DGR_ERR_INVALID_ARG;
    if (!aligned(a, 8) || !aligned(b, 8) || !aligned(sum, 8) || !aligned(prod, 8)) return DGR_ERR_MISALIGNED;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    if (n_pairs == 0) return DGR_OK;
    const int64_t blocks = (n_pairs + 255) / 256;
    packed_ops_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0,
                        static_cast<cudaStream_t>(stream)>>>(reinterpret_cast<const float2 *>(a),
                                                             reinterpret_cast<const float2 *>(b), n_pairs,
                                                             reinterpret_cast<float2 *>(sum),
                                                             reinterpret_cast<float2 *>(prod));
    return launch_status();
}

extern "C" dgr_status dgr_diag_atomic_colsum(const uint16_t *x, int64_t T, int32_t H, float *out, void *stream) {
    if (T < 0 || H < 1 || H > 4096 || !out || (T > 0 && !x) || T > (int64_t{1} << 40)) return DGR_ERR_INVALID_ARG;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(out, 0, static_cast<size_t>(H) * 4, s) != cudaSuccess) return DGR_ERR_CUDA;
    if (T == 0) return DGR_OK;
    const int64_t grid = (T + kAtomicRows - 1) / kAtomicRows;
    if (grid > INT32_MAX) return DGR_ERR_UNSUPPORTED;
    atomic_colsum_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(x, T, H, out);
    return launch_status();
}

extern "C" dgr_status dgr_diag_atomic_rowdot(const uint16_t *dY, const uint16_t *Y, int64_t M, int32_t N,
                                             float *dprob, void *stream) {
    if (M < 0 || N < 1 || N > 65536 || !dprob || (M > 0 && (!dY || !Y)) || M > 65535LL * 8) return DGR_ERR_INVALID_ARG;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(dprob, 0, static_cast<size_t>(M) * 4, s) != cudaSuccess) return DGR_ERR_CUDA;
    if (M == 0) return DGR_OK;
    const dim3 grid(static_cast<unsigned>((N + 127) / 128), static_cast<unsigned>((M + 7) / 8));
    atomic_rowdot_kernel<<<grid, 256, 0, s>>>(dY, Y, M, N, dprob);
    return launch_status();
}

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
