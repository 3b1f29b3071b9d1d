// Grouped dbias: dbias[e][h] = fold_j pw_W(dY[t][h] : t in tile j of expert e).
//
// cuDNN-frontend PR #521, commit "Cover dbias": dbias contends across M-tiles,
// so every (row block, column) gets one FP32 partial with a single writer, and
// a per-expert segment sum reduces the partials in a fixed order, accumulating
// into dbias like the dprob reduction. Expert e owns rows offs[e] ..
// offs[e+1]-1 (device offsets, never read by the host); its tiles are W rows
// counted from its first row.
//
// One persistent launch. A work item is (tile g, block of 32*VE columns):
//   - 8 warps; warp w sums rows [w*W/8, (w+1)*W/8) of the tile in registers
//     (every row's 16-byte load in flight at once), the tree's lower levels;
//   - one thread per column then combines the 8 warp partials by the tree's
//     top three levels (absent row groups pass their sibling up) and writes
//     the tile's slot;
//   - the CTA fences its slots and takes the (expert, column block) ticket;
//     the CTA that takes the expert's last ticket folds the expert's slots in
//     ascending tile order, writes (or adds into) dbias and resets the ticket.
// Integer atomics only count; no floating-point value depends on timing.
#include "dgr_common.cuh"

namespace dgr {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxExperts = 1024;

struct DbiasParams {
    const char *dY;
    int64_t ld;            // elements
    int32_t T, H, E, W;
    int32_t n_cb;          // column blocks of 32 * VE columns
    const int64_t *offs;   // [E + 1], device
    float *out;            // [E, H], row stride ld_out
    int64_t ld_out;
    int32_t accumulate;
    float *slots;          // [tiles, H]
    int32_t *tickets;      // [E, n_cb]
    WsHeader *hdr;
};

__device__ __forceinline__ void unpack(const uint4 &v, float *f, int dtype_bf16) {
    if (dtype_bf16) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
}

// Pairwise tree over the first n (1..L) of L leaves held in v[] (L a power
// of two), in place: v[0] ends as the root. A node whose right child holds no
// present leaf is its left child, unchanged.
template <int L, int VE>
__device__ __forceinline__ void tree_prefix(float (*v)[VE], int n) {
#pragma unroll
    for (int s = 1; s < L; s *= 2) {
#pragma unroll
        for (int i = 0; i + s < L; i += 2 * s)
            if (i + s < n) {
#pragma unroll
                for (int e = 0; e < VE; ++e) v[i][e] = __fadd_rn(v[i][e], v[i + s][e]);
            }
    }
}

// DT_BF16: 1 for bf16 rows (8 a vector), 0 for fp32 (4 a vector). RW: rows a
// warp sums (W / 8).
template <int DT_BF16, int RW>
__global__ void __launch_bounds__(kThreads, 2) dbias_kernel(const DbiasParams p) {
    constexpr int VE = DT_BF16 ? 8 : 4;
    constexpr int CBW = 32 * VE;  // columns of a block
    constexpr int es = DT_BF16 ? 2 : 4;
    __shared__ float red[kWarps][CBW];
    __shared__ int32_t tbase[kMaxExperts + 1];  // first tile of each expert; tbase[E] = tiles
    __shared__ int32_t wsum[kWarps];
    __shared__ int32_t bad, ticket;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;

    // the experts' tile bases (every CTA the same), and the offsets' contract
    if (tid == 0) bad = 0;
    __syncthreads();
    int32_t run = 0;
    for (int e0 = 0; e0 < p.E; e0 += kThreads) {
        const int e = e0 + tid;
        int32_t c = 0;
        if (e < p.E) {
            const int64_t a = p.offs[e], b = p.offs[e + 1];
            if (b < a || (e == 0 && a != 0) || (e == p.E - 1 && b != p.T)) bad = 1;
            else c = static_cast<int32_t>((b - a + p.W - 1) / p.W);
        }
        int32_t incl = c;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, s);
            if (lane >= s) incl += o;
        }
        if (lane == 31) wsum[w] = incl;
        __syncthreads();
        int32_t before = run;
        for (int v = 0; v < w; ++v) before += wsum[v];
        if (e < p.E) tbase[e] = before + incl - c;
        for (int v = 0; v < kWarps; ++v) run += wsum[v];
        __syncthreads();
    }
    if (tid == 0) tbase[p.E] = run;
    __syncthreads();
    if (bad) {
        if (blockIdx.x == 0 && tid == 0) record_error(p.hdr, DGR_ERR_INVALID_ARG, 20);
        return;
    }
    // overwrite: an expert with no rows gets +0.0
    if (blockIdx.x == 0 && !p.accumulate) {
        for (int e = 0; e < p.E; ++e)
            if (tbase[e + 1] == tbase[e])
                for (int h = tid; h < p.H; h += kThreads) p.out[static_cast<int64_t>(e) * p.ld_out + h] = 0.0f;
    }

    const int64_t n_items = static_cast<int64_t>(tbase[p.E]) * p.n_cb;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int32_t g = static_cast<int32_t>(item / p.n_cb);
        const int cb = static_cast<int>(item - static_cast<int64_t>(g) * p.n_cb);
        // expert of tile g: the last e with tbase[e] <= g (empty experts share a base)
        int lo = 0, hi = p.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tbase[mid] <= g) lo = mid;
            else hi = mid - 1;
        }
        const int e = lo;
        const int32_t j = g - tbase[e];
        const int64_t r_first = p.offs[e] + static_cast<int64_t>(j) * p.W;
        const int count = static_cast<int>(min(static_cast<int64_t>(p.W), p.offs[e + 1] - r_first));
        const int col = cb * CBW + lane * VE;
        const bool col_ok = col < p.H;

        // rows [w*RW, w*RW + RW) of the tile: all loads in flight, then the tree
        const int n_here = max(0, min(RW, count - w * RW));
        uint4 raw[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            raw[r] = make_uint4(0u, 0u, 0u, 0u);
            ldg_nc_v4u_if(raw[r], p.dY + ((r_first + w * RW + r) * p.ld + col) * es, col_ok && r < n_here);
        }
        float v[RW][VE];
#pragma unroll
        for (int r = 0; r < RW; ++r) unpack(raw[r], v[r], DT_BF16);
        tree_prefix<RW, VE>(v, n_here);
        if (n_here > 0) {
#pragma unroll
            for (int e2 = 0; e2 < VE; ++e2) red[w][lane * VE + e2] = v[0][e2];
        }
        __syncthreads();
        // top levels across the warps' row groups, one thread per column
        const int nw = (count + RW - 1) / RW;  // row groups present (>= 1)
        const int c = cb * CBW + tid;
        if (tid < CBW && c < p.H) {
            float u[kWarps][1];
#pragma unroll
            for (int q = 0; q < kWarps; ++q) u[q][0] = q < nw ? red[q][tid] : 0.0f;
            tree_prefix<kWarps, 1>(u, nw);
            p.slots[static_cast<int64_t>(g) * p.H + c] = u[0][0];
        }
        __threadfence();  // this thread's slot before the ticket
        __syncthreads();
        const int32_t n_tiles_e = tbase[e + 1] - tbase[e];
        if (tid == 0) ticket = atomicAdd(&p.tickets[e * p.n_cb + cb], 1);
        __syncthreads();
        if (ticket == n_tiles_e - 1) {
            // the expert's last tile of this column block: fold its slots in
            // ascending tile order (every other CTA fenced its slot before
            // its ticket)
            __threadfence();
            if (tid < CBW && c < p.H) {
                const float *s = p.slots + static_cast<int64_t>(tbase[e]) * p.H + c;
                float F = 0.0f;
                for (int j0 = 0; j0 < n_tiles_e; j0 += 16) {
                    float x[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (j0 + u < n_tiles_e) x[u] = __ldcg(s + static_cast<int64_t>(j0 + u) * p.H);
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (j0 + u < n_tiles_e) F = (j0 + u == 0) ? x[u] : __fadd_rn(F, x[u]);
                }
                float *o = p.out + static_cast<int64_t>(e) * p.ld_out + c;
                *o = p.accumulate ? __fadd_rn(*o, F) : F;
            }
            if (tid == 0) p.tickets[e * p.n_cb + cb] = 0;  // ready for the next call
        }
        __syncthreads();  // red[] and ticket are reused by the next item
    }
}

struct DbiasLayout {
    int64_t n_tiles_max;
    int32_t n_cb_max;
    size_t tickets, slots, total;
};

// Tiles: at most ceil(T / W) + E (each expert's last tile may be partial).
// Tickets are sized for the narrower fp32 column blocks (128 columns).
DbiasLayout dbias_layout(int64_t T, int64_t H, int64_t E, int64_t W) {
    DbiasLayout L{};
    L.n_tiles_max = (T + W - 1) / W + E;
    L.n_cb_max = static_cast<int32_t>((H + 127) / 128);
    size_t o = sizeof(WsHeader);
    L.tickets = o;
    o += align_up(static_cast<size_t>(E) * L.n_cb_max * 4);
    L.slots = o;
    o += align_up(static_cast<size_t>(L.n_tiles_max) * H * 4);
    L.total = o;
    return L;
}

template <int DT_BF16, int RW>
dgr_status launch_dbias(const DbiasParams &p, int grid, cudaStream_t s) {
    dbias_kernel<DT_BF16, RW><<<grid, kThreads, 0, s>>>(p);
    return launch_status();
}

template <int DT_BF16>
dgr_status launch_dbias_w(const DbiasParams &p, int grid, cudaStream_t s) {
    switch (p.W) {
        case 8: return launch_dbias<DT_BF16, 1>(p, grid, s);
        case 16: return launch_dbias<DT_BF16, 2>(p, grid, s);
        case 32: return launch_dbias<DT_BF16, 4>(p, grid, s);
        case 64: return launch_dbias<DT_BF16, 8>(p, grid, s);
        case 128: return launch_dbias<DT_BF16, 16>(p, grid, s);
        default: return DGR_ERR_UNSUPPORTED;
    }
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" size_t dgr_dbias_workspace_bytes(int64_t T, int64_t H, int32_t E, int32_t tile_rows) {
    if (T < 0 || H < 0 || H > (1 << 20) || E < 1 || E > kMaxExperts || T > INT32_MAX || !is_pow2(tile_rows) ||
        tile_rows > 128)
        return 0;
    return dbias_layout(T, H, E, tile_rows).total;
}

extern "C" dgr_status dgr_grouped_dbias(const void *dY, int32_t dtype, int64_t T, int64_t H, int64_t ld_dy,
                                        const int64_t *d_offs, int32_t E, float *dbias, int64_t ld_out,
                                        int32_t accumulate, int32_t tile_rows, void *ws, size_t ws_bytes,
                                        void *stream) {
    if (dtype != DGR_DTYPE_BF16 && dtype != DGR_DTYPE_F32) return DGR_ERR_INVALID_ARG;
    if (T < 0 || H < 0 || E < 1 || ld_dy < H || ld_out < H || !is_pow2(tile_rows)) return DGR_ERR_INVALID_ARG;
    if (T > INT32_MAX || E > kMaxExperts || H > (1 << 20) || tile_rows < 8 || tile_rows > 128)
        return DGR_ERR_UNSUPPORTED;
    if (!dbias || !d_offs || (T > 0 && H > 0 && !dY)) return DGR_ERR_INVALID_ARG;
    const int es = dtype == DGR_DTYPE_BF16 ? 2 : 4;
    const int ve = 16 / es;
    if (!aligned(dbias, 4) || !aligned(d_offs, 8)) return DGR_ERR_MISALIGNED;
    if (T > 0 && H > 0 && (!aligned(dY, 16) || (H % ve) != 0 || (ld_dy % ve) != 0)) return DGR_ERR_MISALIGNED;
    const DbiasLayout L = dbias_layout(T, H, E, tile_rows);
    const size_t out_bytes = static_cast<size_t>(((E - 1) * ld_out + H) * 4);
    const size_t dy_bytes = T > 0 ? static_cast<size_t>(((T - 1) * ld_dy + H) * es) : 0;
    if (ranges_overlap(dbias, out_bytes, dY, dy_bytes) || ranges_overlap(dbias, out_bytes, d_offs, (E + 1) * 8))
        return DGR_ERR_ALIAS;
    const bool work = T > 0 && H > 0;
    if (work) {
        if (!ws) return DGR_ERR_INVALID_ARG;
        if (ws_bytes < L.total) return DGR_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(ws, kAlign)) return DGR_ERR_MISALIGNED;
        if (ranges_overlap(dbias, out_bytes, ws, L.total)) return DGR_ERR_ALIAS;
    }
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (H == 0) return DGR_OK;
    if (T == 0) {  // every expert is empty: +0.0 on overwrite, untouched on accumulate
        if (accumulate) return DGR_OK;
        return cudaMemset2DAsync(dbias, ld_out * 4, 0, H * 4, E, s) == cudaSuccess ? DGR_OK : DGR_ERR_CUDA;
    }
    DbiasParams p{};
    p.dY = static_cast<const char *>(dY);
    p.ld = ld_dy;
    p.T = static_cast<int32_t>(T);
    p.H = static_cast<int32_t>(H);
    p.E = E;
    p.W = tile_rows;
    p.n_cb = static_cast<int32_t>((H + 32 * ve - 1) / (32 * ve));
    p.offs = d_offs;
    p.out = dbias;
    p.ld_out = ld_out;
    p.accumulate = accumulate ? 1 : 0;
    char *w = static_cast<char *>(ws);
    p.hdr = reinterpret_cast<WsHeader *>(w);
    p.tickets = reinterpret_cast<int32_t *>(w + L.tickets);
    p.slots = reinterpret_cast<float *>(w + L.slots);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DGR_ERR_CUDA;
    // persistent: two CTAs per SM, never more than the items there can be
    const int64_t items_max = L.n_tiles_max * p.n_cb;
    const int grid = static_cast<int>(items_max < 2LL * sms ? items_max : 2LL * sms);
    return dtype == DGR_DTYPE_BF16 ? launch_dbias_w<1>(p, grid, s) : launch_dbias_w<0>(p, grid, s);
}
