// Ordered per-row dprob: dprob[m] = fold_j pw_128(dY[m][n] * Y[m][n] : n in tile j).
//
// cuDNN-frontend PR #521 (grouped gemm dsrelu deterministic dprob), commit
// "deterministic dprob": one FP32 slot per N-tile so that every (token,
// tile_n) has exactly one writer, slots reduced in a fixed order and the
// result accumulated into dprob. Here one warp owns one row: a lane reads 8
// bf16 (16 bytes) of dY and of Y per step, forms the 8 products (one fp32
// multiply each, rounded on its own), sums them by the first three levels of
// the tile's pairwise tree in registers, and the remaining four levels are
// xor-shuffles at distance 1, 2, 4, 8 (adjacent aligned windows, so the tree
// is exactly the canonical one). Lanes 0-15 then hold tile 2i and lanes 16-31
// tile 2i+1; every lane folds the tile partials in ascending order, so the
// slots never leave the chip unless the caller asks for them.
#include "dgr_common.cuh"

namespace dgr {
namespace {

constexpr int kWarps = 4;
constexpr int kTile = 128;

struct RowdotParams {
    const char *dY;
    const char *Y;
    int64_t ld_dy, ld_y;  // elements
    int32_t M, N;
    int32_t n_tiles;
    float *dprob;
    int32_t accumulate;
    float *slots;         // nullable [M][n_tiles]
    Sched sched;          // which warp takes which row
};

template <int DT>
__device__ __forceinline__ void load8(const char *row, int64_t c0, int32_t N, bool vec, float *f) {
    // 8 consecutive elements starting at column c0; absent ones are not read
    if (DT == DGR_DTYPE_BF16) {
        if (vec && c0 + 8 <= N) {
            const uint4 v = ldg_nc_v4(row + c0 * 2);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] = (c0 + i < N) ? bf16_bits_to_f32(reinterpret_cast<const uint16_t *>(row)[c0 + i]) : 0.0f;
        }
    } else {
        if (vec && c0 + 8 <= N) {
            const uint4 a = ldg_nc_v4(row + c0 * 4);
            const uint4 b = ldg_nc_v4(row + c0 * 4 + 16);
            f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
            f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
            f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
            f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] = (c0 + i < N) ? reinterpret_cast<const float *>(row)[c0 + i] : 0.0f;
        }
    }
}

// Tile partial of the 8-column window of this lane and its 15 neighbours.
__device__ __forceinline__ float lane_tile_partial(const float *a, const float *b, int nvalid, int lane) {
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = __fmul_rn(a[i], b[i]);
    // levels 1-3 in registers over aligned windows, absent columns skipped
#pragma unroll
    for (int s = 1; s < 8; s *= 2) {
#pragma unroll
        for (int r = 0; r + s < 8; r += 2 * s)
            if (r + s < nvalid) p[r] = __fadd_rn(p[r], p[r + s]);
    }
    float v = p[0];
    bool present = nvalid > 0;
    // levels 4-7: partner windows at lane distance 1, 2, 4, 8
#pragma unroll
    for (int s = 1; s < 16; s *= 2) {
        const float o = __shfl_xor_sync(0xffffffffu, v, s);
        const bool o_present = __shfl_xor_sync(0xffffffffu, present ? 1 : 0, s) != 0;
        const bool left_is_me = (lane & s) == 0;
        const bool right_present = left_is_me ? o_present : present;
        const bool left_present = left_is_me ? present : o_present;
        if (left_present && right_present) v = __fadd_rn(v, o);
        else if (!left_is_me && left_present) v = o;  // right absent: the left passes up
        present = left_present;
    }
    return v;
}

// The same when all 256 columns of the step are present: no presence flags.
__device__ __forceinline__ float lane_tile_partial_full(const float *a, const float *b) {
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = __fmul_rn(a[i], b[i]);
    p[0] = __fadd_rn(p[0], p[1]);
    p[2] = __fadd_rn(p[2], p[3]);
    p[4] = __fadd_rn(p[4], p[5]);
    p[6] = __fadd_rn(p[6], p[7]);
    p[0] = __fadd_rn(p[0], p[2]);
    p[4] = __fadd_rn(p[4], p[6]);
    float v = __fadd_rn(p[0], p[4]);
#pragma unroll
    for (int s = 1; s < 16; s *= 2) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, s));
    return v;
}

template <int DT>
__device__ __forceinline__ void unpack_raw(const uint4 *r, float *f) {
    if (DT == DGR_DTYPE_BF16) {
        const uint32_t w[4] = {r[0].x, r[0].y, r[0].z, r[0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
        f[0] = __uint_as_float(r[0].x); f[1] = __uint_as_float(r[0].y);
        f[2] = __uint_as_float(r[0].z); f[3] = __uint_as_float(r[0].w);
        f[4] = __uint_as_float(r[1].x); f[5] = __uint_as_float(r[1].y);
        f[6] = __uint_as_float(r[1].z); f[7] = __uint_as_float(r[1].w);
    }
}

// One row: its tiles' partials and their ordered fold.
template <int DT>
__device__ __forceinline__ void rowdot_row(const RowdotParams &p, int64_t m, int vec, int lane) {
    const int es = DT == DGR_DTYPE_BF16 ? 2 : 4;
    const char *rdy = p.dY + m * p.ld_dy * es;
    const char *ry = p.Y + m * p.ld_y * es;
    // raw 16-byte words stay in flight (U steps per lane) and are widened at use
    constexpr int V = DT == DGR_DTYPE_BF16 ? 1 : 2;  // uint4 per 8 elements
    constexpr int U = DT == DGR_DTYPE_BF16 ? 8 : 4;  // 256-column steps in flight per lane
    float F = 0.0f;
    const int n_steps = (p.N + 255) / 256;  // each step covers two tiles
    for (int i0 = 0; i0 < n_steps; i0 += U) {
        uint4 ra[U][V], rb[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c0 = static_cast<int64_t>(i0 + u) * 256 + lane * 8;
            if (vec && i0 + u < n_steps && c0 + 8 <= p.N) {
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    ra[u][q] = ldg_nc_v4(rdy + c0 * es + 16 * q);
                    rb[u][q] = ldg_nc_v4(ry + c0 * es + 16 * q);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u;
            if (i >= n_steps) break;
            const int64_t c0 = static_cast<int64_t>(i) * 256 + lane * 8;
            float a[8], b[8];
            if (vec && c0 + 8 <= p.N) {
                unpack_raw<DT>(ra[u], a);
                unpack_raw<DT>(rb[u], b);
            } else if (c0 < p.N) {
                load8<DT>(rdy, c0, p.N, false, a);
                load8<DT>(ry, c0, p.N, false, b);
            }
            float v;
            if (static_cast<int64_t>(i) * 256 + 256 <= p.N) {
                v = lane_tile_partial_full(a, b);
            } else {
                const int nvalid = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(8), p.N - c0)));
                v = lane_tile_partial(a, b, nvalid, lane);
            }
            const float t0 = __shfl_sync(0xffffffffu, v, 0);
            const float t1 = __shfl_sync(0xffffffffu, v, 16);
            const int j0 = 2 * i, j1 = 2 * i + 1;
            F = (j0 == 0) ? t0 : __fadd_rn(F, t0);
            if (j1 < p.n_tiles) F = __fadd_rn(F, t1);
            if (p.slots && lane == 0) {
                p.slots[m * p.n_tiles + j0] = t0;
                if (j1 < p.n_tiles) p.slots[m * p.n_tiles + j1] = t1;
            }
        }
    }
    if (lane == 0) p.dprob[m] = p.accumulate ? __fadd_rn(p.dprob[m], F) : F;
}

// One warp per row (rows handed out in the schedule's order; with a capped
// grid a warp takes several).
template <int DT>
__global__ void __launch_bounds__(kWarps * 32) rowdot_kernel(const RowdotParams p, int vec) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); i < p.M; i += nw)
        rowdot_row<DT>(p, sched_item(p.sched, static_cast<uint32_t>(i)), vec, lane);
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" size_t dgr_rowdot_workspace_bytes(int64_t M, int64_t N, int32_t tile_n) {
    (void)M;
    (void)N;
    (void)tile_n;
    return 0;  // the fold stays in registers
}

extern "C" dgr_status dgr_ordered_rowdot_dprob(const void *dY, const void *Y, int32_t dtype, int64_t M,
                                               int64_t N, int64_t ld_dy, int64_t ld_y, float *dprob,
                                               int32_t accumulate, int32_t tile_n, float *slots, void *ws,
                                               size_t ws_bytes, void *stream) {
    (void)ws;
    (void)ws_bytes;
    if (dtype != DGR_DTYPE_BF16 && dtype != DGR_DTYPE_F32) return DGR_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || tile_n != kTile) return DGR_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > 65536) return DGR_ERR_UNSUPPORTED;
    if (M == 0) return DGR_OK;
    if (!dprob || (N > 0 && (!dY || !Y))) return DGR_ERR_INVALID_ARG;
    if (ld_dy < N || ld_y < N) return DGR_ERR_INVALID_ARG;
    const int es = dtype == DGR_DTYPE_BF16 ? 2 : 4;
    if (!aligned(dprob, 4) || !aligned(dY, es) || !aligned(Y, es) || (slots && !aligned(slots, 4)))
        return DGR_ERR_MISALIGNED;
    const int64_t n_tiles = (N + kTile - 1) / kTile;
    const size_t ext_dy = N > 0 ? static_cast<size_t>(((M - 1) * ld_dy + N) * es) : 0;
    const size_t ext_y = N > 0 ? static_cast<size_t>(((M - 1) * ld_y + N) * es) : 0;
    const size_t ext_slots = slots ? static_cast<size_t>(M * n_tiles * 4) : 0;
    if (ranges_overlap(dprob, M * 4, dY, ext_dy) || ranges_overlap(dprob, M * 4, Y, ext_y) ||
        ranges_overlap(slots, ext_slots, dY, ext_dy) || ranges_overlap(slots, ext_slots, Y, ext_y) ||
        ranges_overlap(slots, ext_slots, dprob, M * 4))
        return DGR_ERR_ALIAS;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        if (accumulate) return DGR_OK;
        return cudaMemsetAsync(dprob, 0, M * 4, s) == cudaSuccess ? DGR_OK : DGR_ERR_CUDA;
    }
    RowdotParams p{};
    p.dY = static_cast<const char *>(dY);
    p.Y = static_cast<const char *>(Y);
    p.ld_dy = ld_dy;
    p.ld_y = ld_y;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.n_tiles = static_cast<int32_t>(n_tiles);
    p.dprob = dprob;
    p.accumulate = accumulate ? 1 : 0;
    p.slots = slots;
    const int vec = (aligned(dY, 16) && aligned(Y, 16) && (ld_dy * es) % 16 == 0 && (ld_y * es) % 16 == 0) ? 1 : 0;
    p.sched = sched_for(static_cast<uint32_t>(M));
    const unsigned grid = sched_grid(static_cast<unsigned>((M + kWarps - 1) / kWarps));
    if (dtype == DGR_DTYPE_BF16)
        rowdot_kernel<DGR_DTYPE_BF16><<<grid, kWarps * 32, 0, s>>>(p, vec);
    else
        rowdot_kernel<DGR_DTYPE_F32><<<grid, kWarps * 32, 0, s>>>(p, vec);
    return launch_status();
}
