// Grouped dbias: dbias[e][h] = fold_j pw_W(dY[t][h] : t in tile j of expert e).
//
// cuDNN-frontend PR #521, commit "Cover dbias": dbias contends across M-tiles,
// so every (row block, column) gets one FP32 partial with a single writer, and
// a per-expert segment sum reduces the partials in a fixed order, accumulating
// into dbias like the dprob reduction. Expert e owns rows offs[e] ..
// offs[e+1]-1 (device offsets, never read by the host); its tiles are W rows
// counted from its first row.
//
// Two launches:
//   produce - persistent, one CTA of 16 warps per SM. A work item is (tile g,
//             block of V 16-byte column vectors) and belongs to one warp:
//             lane = (row group, vector), 32 / V row groups of consecutive
//             rows. A lane sums its rows by the tile tree's lower levels in
//             registers, 16 rows' loads in flight at a time (batches are
//             aligned subtrees, combined through a binary-counter stack); the
//             upper levels are xor-shuffles between row groups; row group 0
//             stores the item's partials. No barrier, no fence, no atomic.
//   fold    - one thread per (expert, column), started early by programmatic
//             dependent launch and waiting for the producers' grid: the
//             expert's partials folded in ascending tile order, then written
//             or added to dbias with one rounding; an expert with no rows
//             gets +0.0 on overwrite.
// No floating-point value depends on timing.
#include "dgr_common.cuh"

namespace dgr {
namespace {

constexpr int kProdThreads = 512;
constexpr int kProdWarps = kProdThreads / 32;
constexpr int kFoldThreads = 256;
constexpr int kMaxExperts = 1024;

struct DbiasParams {
    const char *dY;
    int64_t ld;            // elements
    int32_t T, H, E, W;
    int32_t n_cb;          // column blocks of V * VE columns
    const int64_t *offs;   // [E + 1], device
    float *out;            // [E, H], row stride ld_out
    int64_t ld_out;
    int32_t accumulate;
    float *slots;          // [tiles, H]
    WsHeader *hdr;
};

__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// tbase[e] = first tile of expert e (tbase[E] = all tiles), from the device
// offsets, by the whole block (every block computes the same). Returns false
// when the offsets break the contract (decreasing, offs[0] != 0, offs[E] != T).
__device__ bool tile_bases(const DbiasParams &p, int32_t *tbase, int64_t *soffs, int32_t *wsum, int32_t *bad) {
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, nt = blockDim.x, nw = nt >> 5;
    if (tid == 0) *bad = 0;
    __syncthreads();
    int32_t run = 0;
    for (int e0 = 0; e0 < p.E; e0 += nt) {
        const int e = e0 + tid;
        int32_t c = 0;
        if (e < p.E) {
            const int64_t a = p.offs[e], b = p.offs[e + 1];
            soffs[e] = a;
            if (e == p.E - 1) soffs[p.E] = b;
            if (b < a || (e == 0 && a != 0) || (e == p.E - 1 && b != p.T)) *bad = 1;
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
        for (int v = 0; v < nw; ++v) run += wsum[v];
        __syncthreads();
    }
    if (tid == 0) tbase[p.E] = run;
    __syncthreads();
    return *bad == 0;
}


// The same predicated 16-byte load with a 256-byte L2 fetch: a 128-byte
// access brings its neighbour (the next item's columns) with it.
__device__ __forceinline__ void ldg_v4u_l2_256_if(uint4 &v, const void *ptr, bool pred) {
    asm volatile(
        "{ .reg .pred q; setp.ne.b32 q, %5, 0;\n\t"
        "@q ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4]; }"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
        : "l"(ptr), "r"(static_cast<int>(pred)));
}

template <int DT_BF16>
__device__ __forceinline__ void unpack(const uint4 &v, float *f) {
    if (DT_BF16) {
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

// 16-byte column vectors of an item (a warp): 8 row groups of W / 8 rows.
// Measured on the 65536 x 2048 workload: 8 vectors (4 row groups) 71.6 us,
// 4 vectors 56.4 us, 2 vectors 70.0 us; narrow items give many small units
// of work, each a short chain of loads.
constexpr int kItemVectors = 4;

// DT_BF16: 1 for bf16 rows (8 a vector), 0 for fp32 (4 a vector); W: tile
// rows; V: column vectors of an item.
template <int DT_BF16, int W, int V>
__global__ void __launch_bounds__(kProdThreads, 1) dbias_produce(const DbiasParams p) {
    constexpr int VE = DT_BF16 ? 8 : 4;
    constexpr int CBW = V * VE;                  // columns of a block
    constexpr int es = DT_BF16 ? 2 : 4;
    constexpr int RGW = 32 / V;                  // row groups
    constexpr int RPL = W / RGW;                 // rows a lane
    static_assert(RPL >= 1, "a row a lane at least");
    constexpr int BATCH = RPL < 16 ? RPL : 16;   // rows in flight a lane
    constexpr int NB = RPL / BATCH;              // batches, a power of two <= 16
    constexpr int LV = NB >= 16 ? 4 : NB >= 8 ? 3 : NB >= 4 ? 2 : NB >= 2 ? 1 : 0;
    __shared__ int32_t tbase[kMaxExperts + 1];
    __shared__ int64_t soffs[kMaxExperts + 1];  // the offsets, read once
    __shared__ int32_t wsum[kProdWarps];
    __shared__ int32_t bad;
    launch_dependents();  // the fold launch may start its blocks; it waits for this grid
    if (!tile_bases(p, tbase, soffs, wsum, &bad)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(p.hdr, DGR_ERR_INVALID_ARG, 20);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t n_items = static_cast<int64_t>(tbase[p.E]) * p.n_cb;
    const int64_t n_warps = static_cast<int64_t>(gridDim.x) * kProdWarps;
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * kProdWarps + (threadIdx.x >> 5); item < n_items;
         item += n_warps) {
        const int32_t g = static_cast<int32_t>(item / p.n_cb);
        const int cb = static_cast<int>(item - static_cast<int64_t>(g) * p.n_cb);
        // expert of tile g: the last e with tbase[e] <= g (empty experts share a base)
        int lo = 0, hi = p.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tbase[mid] <= g) lo = mid;
            else hi = mid - 1;
        }
        const int64_t r_first = soffs[lo] + static_cast<int64_t>(g - tbase[lo]) * W;
        const int count = static_cast<int>(min(static_cast<int64_t>(W), soffs[lo + 1] - r_first));
        const int rg = lane / V;
        const int col = cb * CBW + (lane - rg * V) * VE;
        const bool col_ok = col < p.H;
        const int nrows = max(0, min(RPL, count - rg * RPL));  // this lane's rows present
        const char *src = p.dY + ((r_first + rg * RPL) * p.ld + col) * es;
        float stack[LV + 1][VE];
        float acc[VE];
#pragma unroll
        for (int bi = 0; bi < NB; ++bi) {
            const int rb = bi * BATCH;
            uint4 raw[BATCH];
#pragma unroll
            for (int r = 0; r < BATCH; ++r) {
                raw[r] = make_uint4(0u, 0u, 0u, 0u);
                ldg_v4u_l2_256_if(raw[r], src + static_cast<int64_t>(rb + r) * p.ld * es, col_ok && rb + r < nrows);
            }
            // the batch's subtree (rows rb .. rb+BATCH-1), absent rows skipped;
            // level 1 is taken while widening, pair by pair
            const int nb_rows = max(0, min(BATCH, nrows - rb));
            constexpr int NP = BATCH > 1 ? BATCH / 2 : 1;
            float lv[NP][VE];
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                unpack<DT_BF16>(raw[2 * i], lv[i]);
                if (BATCH > 1 && 2 * i + 1 < nb_rows) {
                    float b2[VE];
                    unpack<DT_BF16>(raw[2 * i + 1], b2);
                    vadd<VE>(lv[i], lv[i], b2);
                }
            }
            const int np_present = (nb_rows + 1) / 2;
#pragma unroll
            for (int sft = 1; sft < NP; sft *= 2) {
#pragma unroll
                for (int i = 0; i + sft < NP; i += 2 * sft)
                    if (i + sft < np_present) vadd<VE>(lv[i], lv[i], lv[i + sft]);
            }
            // push batch bi (a compile-time index) onto the binary-counter stack
            if (nb_rows > 0) {
#pragma unroll
                for (int e = 0; e < VE; ++e) acc[e] = lv[0][e];
                int lvl = 0;
#pragma unroll
                for (int l = 0; l < LV; ++l) {
                    if (((bi >> l) & 1) == 0) break;
                    vadd<VE>(acc, stack[l], acc);
                    lvl = l + 1;
                }
#pragma unroll
                for (int l = 0; l <= LV; ++l)
                    if (l == lvl) {
#pragma unroll
                        for (int e = 0; e < VE; ++e) stack[l][e] = acc[e];
                    }
            }
        }
        // ragged end: complete blocks of the set bits of the present batch
        // count, smallest first, each larger (earlier) block on the left
        const int nbp = (nrows + BATCH - 1) / BATCH;
        bool have = false;
#pragma unroll
        for (int l = 0; l <= LV; ++l) {
            if ((nbp >> l) & 1) {
#pragma unroll
                for (int e = 0; e < VE; ++e) acc[e] = have ? __fadd_rn(stack[l][e], acc[e]) : stack[l][e];
                have = true;
            }
        }
        // upper levels: row group q absorbs q + s (lane distance s * V)
        bool present = nrows > 0;
#pragma unroll
        for (int s = 1; s < RGW; s *= 2) {
            const bool left_is_me = (rg & s) == 0;
            const bool o_present = __shfl_xor_sync(0xffffffffu, present ? 1 : 0, s * V) != 0;
            const bool left_present = left_is_me ? present : o_present;
            const bool right_present = left_is_me ? o_present : present;
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                const float o = __shfl_xor_sync(0xffffffffu, acc[e], s * V);
                if (left_present && right_present) acc[e] = __fadd_rn(acc[e], o);
                else if (!left_is_me && left_present) acc[e] = o;
            }
            present = left_present;
        }
        if (rg == 0 && col_ok) {
            float4 *dst = reinterpret_cast<float4 *>(p.slots + static_cast<int64_t>(g) * p.H + col);
#pragma unroll
            for (int q = 0; q < VE / 4; ++q)
                dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        }
    }
}

__global__ void __launch_bounds__(kFoldThreads) dbias_fold(const DbiasParams p) {
    __shared__ int32_t tbase[kMaxExperts + 1];
    __shared__ int64_t soffs[kMaxExperts + 1];
    __shared__ int32_t wsum[kFoldThreads / 32];
    __shared__ int32_t bad;
    const bool ok = tile_bases(p, tbase, soffs, wsum, &bad);  // the offsets only: no producer output yet
    grid_dep_wait();  // the producers' grid has completed and its partials are visible
    if (!ok) return;  // the producers recorded the error
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kFoldThreads + threadIdx.x;
    if (i >= static_cast<int64_t>(p.E) * p.H) return;
    const int e = static_cast<int>(i / p.H);
    const int h = static_cast<int>(i - static_cast<int64_t>(e) * p.H);
    const int32_t n = tbase[e + 1] - tbase[e];
    float *o = p.out + static_cast<int64_t>(e) * p.ld_out + h;
    if (n == 0) {
        if (!p.accumulate) *o = 0.0f;
        return;
    }
    const float *s = p.slots + static_cast<int64_t>(tbase[e]) * p.H + h;
    float F = 0.0f;
    for (int j0 = 0; j0 < n; j0 += 32) {
        float x[32];
#pragma unroll
        for (int u = 0; u < 32; ++u)
            if (j0 + u < n) x[u] = __ldcg(s + static_cast<int64_t>(j0 + u) * p.H);
#pragma unroll
        for (int u = 0; u < 32; ++u)
            if (j0 + u < n) F = (j0 + u == 0) ? x[u] : __fadd_rn(F, x[u]);
    }
    *o = p.accumulate ? __fadd_rn(*o, F) : F;
}

struct DbiasLayout {
    int64_t n_tiles_max;
    size_t slots, total;
};

// Tiles: at most ceil(T / W) + E (each expert's last tile may be partial).
DbiasLayout dbias_layout(int64_t T, int64_t H, int64_t E, int64_t W) {
    DbiasLayout L{};
    L.n_tiles_max = (T + W - 1) / W + E;
    L.slots = sizeof(WsHeader);
    L.total = L.slots + align_up(static_cast<size_t>(L.n_tiles_max) * H * 4);
    return L;
}

template <int DT_BF16>
dgr_status launch_produce(const DbiasParams &p, int grid, cudaStream_t s) {
    switch (p.W) {
        case 8: dbias_produce<DT_BF16, 8, kItemVectors><<<grid, kProdThreads, 0, s>>>(p); break;
        case 16: dbias_produce<DT_BF16, 16, kItemVectors><<<grid, kProdThreads, 0, s>>>(p); break;
        case 32: dbias_produce<DT_BF16, 32, kItemVectors><<<grid, kProdThreads, 0, s>>>(p); break;
        case 64: dbias_produce<DT_BF16, 64, kItemVectors><<<grid, kProdThreads, 0, s>>>(p); break;
        case 128: dbias_produce<DT_BF16, 128, kItemVectors><<<grid, kProdThreads, 0, s>>>(p); break;
        default: return DGR_ERR_UNSUPPORTED;
    }
    return launch_status();
}

// The fold may start its blocks while the producers finish (it computes the
// tile bases from the offsets first) and reads the partials only after
// griddepcontrol.wait.
dgr_status launch_fold(const DbiasParams &p, cudaStream_t s) {
    const int64_t n = static_cast<int64_t>(p.E) * p.H;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>((n + kFoldThreads - 1) / kFoldThreads));
    cfg.blockDim = dim3(kFoldThreads);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dbias_fold, p) == cudaSuccess ? DGR_OK : DGR_ERR_CUDA;
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
    p.n_cb = static_cast<int32_t>((H + kItemVectors * ve - 1) / (kItemVectors * ve));
    p.offs = d_offs;
    p.out = dbias;
    p.ld_out = ld_out;
    p.accumulate = accumulate ? 1 : 0;
    char *w = static_cast<char *>(ws);
    p.hdr = reinterpret_cast<WsHeader *>(w);
    p.slots = reinterpret_cast<float *>(w + L.slots);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DGR_ERR_CUDA;
    // producers: one 16-warp CTA per SM, never more than the items need
    const int64_t items_max = L.n_tiles_max * p.n_cb;
    const int64_t want = (items_max + kProdWarps - 1) / kProdWarps;
    const int grid = static_cast<int>(want < sms ? want : sms);
    st = dtype == DGR_DTYPE_BF16 ? launch_produce<1>(p, grid, s) : launch_produce<0>(p, grid, s);
    if (st != DGR_OK) return st;
    return launch_fold(p, s);
}
