// Deterministic index_add: stable radix sort by destination, then segmented
// pairwise sums in original order, padding routed to the dummy row R.
//
// Megatron-LM PR #7441 (DSv4 --deterministic-mode), Source 3: the atomic-free
// dK is an index_add done as a stable sort plus a (prefix) sum, with padding
// slots spread over dummy rows that the caller drops. Four launches:
//   K1 count   - map idx to keys (idx outside [0, R) -> R; outside [-1, R) is
//                counted), per-block histograms of the key's high byte and each
//                bucket's key range; the last block to finish scans the
//                histograms (digit-major) into per-block scatter offsets and
//                bucket starts, and marks buckets that hold a single key.
//   K2 scatter - stable scatter by the high byte: inside a block, elements are
//                ranked in original order with warp match/ballot and per-warp
//                digit counters, so equal digits keep their input order. A
//                single-key bucket (the dummy row) is already in final order
//                and goes straight to the sorted arrays.
//   K3 bucket  - one block per high-byte bucket: counting sort by the low byte
//                (stable, same ranking), which also yields seg_start[] for the
//                bucket's 256 keys, and lists the tiles of rows too long for
//                one warp.
//   K4 segsum  - one warp per destination row sums its members (in original
//                order) by the pairwise tree over tiles of 128 members and folds
//                the tiles in order, then out[r] += sum with one rounding.
//                Rows with more than 8 tiles are split: one warp per 32-member
//                quarter of each listed tile writes a slot; the last quarter of a tile
//                to arrive (an integer ticket) combines the quarters into the
//                tile partial, and the last tile of the row folds the tile
//                partials in order.
// Integer atomics only count; no floating-point value depends on timing.
#include "dgr_common.cuh"

namespace dgr {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 32;
constexpr int kBlockElems = kThreads * kItems;  // 8192 elements per sort block
constexpr int kDigits = 256;
constexpr int kSegTile = 128;
constexpr int kWarpMaxTiles = 8;                // rows up to 1024 members: one warp
constexpr int kSub = 32;                         // split-row work unit (a quarter tile)
constexpr int kStackLevels = 5;                  // group stack depth for 16 groups of 8

struct IdxParams {
    const int32_t *idx;
    int32_t N, R, D;
    int32_t nb;             // sort blocks
    int32_t n_buckets;      // high-byte buckets covering keys 0..R
    int32_t n_pblk;         // 128-position blocks of the sorted order (slot indexing)
    int32_t seg_tile;
    const float *src;
    int64_t ld_src;
    float *out;
    int64_t ld_out;
    int32_t *bad_count;
    int32_t *keys_a, *vals_a, *perm, *skey, *hist, *offs, *bucket_start, *seg_start, *tickets, *tile_tickets;
    int32_t *bucket_negmin, *bucket_max, *bucket_key;
    int2 *heavy;  // (row, tile) of every tile of a row with more than 8 tiles
    float *slots;
    WsHeader *hdr;
};

__device__ __forceinline__ int32_t map_key(int32_t v, int32_t R, bool &bad) {
    if (v >= 0 && v < R) return v;
    bad = (v != -1);
    return R;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---------------------------------------------------------------------------
// K1: high-byte histograms per block; the last block scans them.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) count_kernel(const IdxParams p) {
    __shared__ int32_t h[kDigits];
    __shared__ int32_t mn[kDigits];
    __shared__ int32_t mx[kDigits];
    __shared__ int32_t base[kDigits + 1];
    __shared__ int32_t bad_block;
    __shared__ int is_last;
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    h[tid] = 0;
    mn[tid] = INT32_MAX;
    mx[tid] = -1;
    if (tid == 0) bad_block = 0;
    if (b == 0 && tid == 0) p.hdr->pad[3] = 0;  // heavy-tile list of this call starts empty
    __syncthreads();
    int32_t v[kItems];
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const int64_t e = static_cast<int64_t>(b) * kBlockElems + r * kThreads + tid;
        v[r] = e < p.N ? p.idx[e] : INT32_MIN;
    }
    int my_bad = 0;
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        if (v[r] == INT32_MIN && static_cast<int64_t>(b) * kBlockElems + r * kThreads + tid >= p.N) continue;
        bool bad = false;
        const int32_t k = map_key(v[r], p.R, bad);
        my_bad += bad ? 1 : 0;
        atomicAdd(&h[k >> 8], 1);
        atomicMin(&mn[k >> 8], k);
        atomicMax(&mx[k >> 8], k);
    }
    if (my_bad) atomicAdd(&bad_block, my_bad);
    __syncthreads();
    p.hist[static_cast<int64_t>(b) * kDigits + tid] = h[tid];
    if (h[tid] > 0) {
        // per-bucket key range over all blocks (integer max: order-free)
        atomicMax(&p.bucket_negmin[tid], INT32_MAX - mn[tid]);
        atomicMax(&p.bucket_max[tid], mx[tid]);
    }
    if (tid == 0 && bad_block) atomicAdd(&p.hdr->pad[2], bad_block);
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(&p.hdr->pad[1], 1) == p.nb - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // digit-major exclusive scan: offs[b][d] = sum of digits < d + counts of d in blocks < b
    int32_t total = 0;
    for (int b0 = 0; b0 < p.nb; b0 += 16) {
        int32_t c[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
            c[u] = (b0 + u < p.nb) ? __ldcg(&p.hist[static_cast<int64_t>(b0 + u) * kDigits + tid]) : 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) total += c[u];
    }
    h[tid] = total;
    __syncthreads();
    if (tid == 0) {
        int32_t run = 0;
        for (int d = 0; d < kDigits; ++d) {
            base[d] = run;
            run += h[d];
        }
        base[kDigits] = run;
    }
    __syncthreads();
    int32_t run = base[tid];
    for (int b0 = 0; b0 < p.nb; b0 += 16) {
        int32_t c[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
            c[u] = (b0 + u < p.nb) ? __ldcg(&p.hist[static_cast<int64_t>(b0 + u) * kDigits + tid]) : 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (b0 + u < p.nb) {
                p.offs[static_cast<int64_t>(b0 + u) * kDigits + tid] = run;
                run += c[u];
            }
        }
    }
    p.bucket_start[tid] = base[tid];
    const int32_t kmax = __ldcg(&p.bucket_max[tid]);
    const int32_t kmin = INT32_MAX - __ldcg(&p.bucket_negmin[tid]);
    p.bucket_key[tid] = (total > 0 && kmin == kmax) ? kmax : -1;  // one key: its order is final after K2
    p.bucket_negmin[tid] = 0;
    p.bucket_max[tid] = 0;
    if (tid == 0) {
        p.bucket_start[kDigits] = base[kDigits];
        const int32_t bad = atomicAdd(&p.hdr->pad[2], 0);
        if (p.bad_count) *p.bad_count = bad;
        p.hdr->pad[2] = 0;
        p.hdr->pad[1] = 0;
    }
}

// Stable in-block ranking: warp w owns elements [w*kWarpElems, ...) of the
// block in rounds of 32 (round-major, lane order = element order). Returns
// each element's rank among equal digits inside its warp; cnt[w][d] ends as
// the warp's digit counts.
__device__ __forceinline__ void warp_rank(int digit, bool valid, int32_t (*cnt)[kDigits], int w, int32_t &rank) {
    const int d = valid ? digit : kDigits;  // invalid lanes match each other only
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const int before = __popc(peers & lanemask_lt());
    const int32_t base = valid ? cnt[w][d] : 0;
    __syncwarp();
    if (valid && before == 0) cnt[w][d] = base + __popc(peers);
    __syncwarp();
    rank = base + before;
}

// ---------------------------------------------------------------------------
// K2: stable scatter by the high byte. Elements of a one-key bucket go
// straight to their final place (perm/skey); the others to keys_a/vals_a.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) scatter_high_kernel(const IdxParams p) {
    __shared__ int32_t cnt[kWarps][kDigits];
    __shared__ int32_t pre[kWarps][kDigits];
    __shared__ int32_t boff[kDigits];
    __shared__ int32_t bkey[kDigits];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x;
    for (int q = tid; q < kWarps * kDigits; q += kThreads) (&cnt[0][0])[q] = 0;
    boff[tid] = p.offs[static_cast<int64_t>(b) * kDigits + tid];
    bkey[tid] = p.bucket_key[tid];
    __syncthreads();
    const int64_t e0 = static_cast<int64_t>(b) * kBlockElems + w * (kItems * 32) + lane;
    int32_t key[kItems];
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const int64_t e = e0 + r * 32;
        bool bad = false;
        key[r] = e < p.N ? map_key(p.idx[e], p.R, bad) : -1;
    }
    int32_t rank[kItems];
#pragma unroll
    for (int r = 0; r < kItems; ++r) warp_rank(key[r] >> 8, key[r] >= 0, cnt, w, rank[r]);
    __syncthreads();
    {
        int32_t run = 0;
        for (int ww = 0; ww < kWarps; ++ww) {
            pre[ww][tid] = run;
            run += cnt[ww][tid];
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        if (key[r] < 0) continue;
        const int d = key[r] >> 8;
        const int32_t pos = boff[d] + pre[w][d] + rank[r];
        const int32_t e = static_cast<int32_t>(e0 + r * 32);
        if (bkey[d] >= 0) {
            p.perm[pos] = e;
            p.skey[pos] = key[r];
        } else {
            p.keys_a[pos] = key[r];
            p.vals_a[pos] = e;
        }
    }
}

// Heavy rows (more than kWarpMaxTiles tiles) get one list entry per tile.
__device__ __forceinline__ void list_heavy_tiles(const IdxParams &p, int32_t key, int32_t n) {
    if (n <= kWarpMaxTiles * kSegTile) return;
    const int32_t n_tiles = (n + kSegTile - 1) / kSegTile;
    const int32_t at = atomicAdd(&p.hdr->pad[3], n_tiles);
    for (int32_t t = 0; t < n_tiles; ++t) p.heavy[at + t] = make_int2(key, t);
}

// ---------------------------------------------------------------------------
// K3: per bucket, stable counting sort by the low byte, and segment starts.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) bucket_kernel(const IdxParams p) {
    __shared__ int32_t h[kDigits];
    __shared__ int32_t base[kDigits];
    __shared__ int32_t cnt[kWarps][kDigits];
    __shared__ int32_t pre[kWarps][kDigits];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int d = blockIdx.x;
    const int32_t bs = p.bucket_start[d];
    const int32_t be = p.bucket_start[d + 1];
    const int32_t k = d * 256 + tid;
    const int32_t one_key = p.bucket_key[d];
    if (one_key >= 0) {  // K2 already placed it; only the segment starts remain
        if (k <= p.R) p.seg_start[k] = k <= one_key ? bs : be;
        if (k == p.R) p.seg_start[p.R + 1] = p.N;
        if (tid == 0 && p.seg_tile == kSegTile) list_heavy_tiles(p, one_key, be - bs);
        return;
    }
    h[tid] = 0;
    __syncthreads();
    for (int32_t c0 = bs; c0 < be; c0 += kBlockElems) {
        int32_t kk[kItems];
#pragma unroll
        for (int r = 0; r < kItems; ++r) {
            const int32_t i = c0 + r * kThreads + tid;
            kk[r] = i < be ? p.keys_a[i] : -1;
        }
#pragma unroll
        for (int r = 0; r < kItems; ++r)
            if (kk[r] >= 0) atomicAdd(&h[kk[r] & 255], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int32_t run = 0;
        for (int q = 0; q < kDigits; ++q) {
            base[q] = bs + run;
            run += h[q];
        }
    }
    __syncthreads();
    if (k <= p.R) p.seg_start[k] = base[tid];
    if (k == p.R) p.seg_start[p.R + 1] = p.N;
    if (k <= p.R && p.seg_tile == kSegTile) list_heavy_tiles(p, k, h[tid]);
    for (int32_t c0 = bs; c0 < be; c0 += kBlockElems) {
        for (int q = tid; q < kWarps * kDigits; q += kThreads) (&cnt[0][0])[q] = 0;
        __syncthreads();
        const int32_t e0 = c0 + w * (kItems * 32) + lane;
        int32_t key[kItems], val[kItems], rank[kItems];
#pragma unroll
        for (int r = 0; r < kItems; ++r) {
            const int32_t e = e0 + r * 32;
            key[r] = e < be ? p.keys_a[e] : -1;
            val[r] = e < be ? p.vals_a[e] : 0;
        }
#pragma unroll
        for (int r = 0; r < kItems; ++r) warp_rank(key[r] & 255, key[r] >= 0, cnt, w, rank[r]);
        __syncthreads();
        {
            int32_t run = 0;
            for (int ww = 0; ww < kWarps; ++ww) {
                pre[ww][tid] = run;
                run += cnt[ww][tid];
            }
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kItems; ++r) {
            if (key[r] < 0) continue;
            const int lo = key[r] & 255;
            const int32_t pos = base[lo] + pre[w][lo] + rank[r];
            p.perm[pos] = val[r];
            p.skey[pos] = key[r];
        }
        __syncthreads();
        {
            int32_t add = 0;
            for (int ww = 0; ww < kWarps; ++ww) add += cnt[ww][tid];
            base[tid] += add;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// K4: segmented sums.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float4 f4add(float4 a, float4 b) {
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

__device__ __forceinline__ float4 ld_src4(const IdxParams &p, int32_t row, int col) {
    const uint4 u = ldg_nc_v4(p.src + static_cast<int64_t>(row) * p.ld_src + col);
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}

// Pairwise tree over the members [q0, q0 + cnt) of a window of 8..128
// members (cnt <= 128), in sorted-position order (= original order within a
// row). The window's width does not matter: leaves past cnt are absent, and
// an absent right half passes its left half up unchanged. Each lane sums its 4 columns starting at `col` (col < 0: the
// lane only joins the shuffles). Groups of 8 members are summed in registers;
// a binary-counter stack over groups (in this warp's shared-memory rows `stk`)
// gives the higher levels; absent members (past cnt) are skipped, which is the
// canonical tail rule.
__device__ __forceinline__ float4 window_sum(const IdxParams &p, int32_t q0, int cnt, int col, int lane,
                                          float4 (*stk)[32]) {
    constexpr int kM = kSegTile / 32;
    int32_t pidx[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) {
        const int j = m * 32 + lane;
        pidx[m] = (j < cnt) ? p.perm[q0 + j] : 0;
    }
    const int n_groups = (cnt + 7) / 8;
#pragma unroll 1
    for (int gi = 0; gi < n_groups; ++gi) {
        int32_t mine = pidx[0];
#pragma unroll
        for (int m = 1; m < kM; ++m)
            if ((gi >> 2) == m) mine = pidx[m];
        float4 v[8];
        const int nu = min(8, cnt - gi * 8);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t row = __shfl_sync(0xffffffffu, mine, (gi & 3) * 8 + u);
            if (u < nu && col >= 0) v[u] = ld_src4(p, row, col);
        }
#pragma unroll
        for (int s = 1; s < 8; s *= 2) {
#pragma unroll
            for (int r = 0; r + s < 8; r += 2 * s)
                if (r + s < nu) v[r] = f4add(v[r], v[r + s]);
        }
        // push group gi: carry through the levels where gi has a one bit
        float4 cur = v[0];
        int l = 0;
        while ((gi >> l) & 1) {
            cur = f4add(stk[l][lane], cur);
            ++l;
        }
        stk[l][lane] = cur;
    }
    // ragged end: combine the complete blocks of the set bits of n_groups,
    // smallest first, each larger (earlier) block on the left
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool have = false;
    for (int l = 0; (n_groups >> l) != 0; ++l) {
        if ((n_groups >> l) & 1) {
            acc = have ? f4add(stk[l][lane], acc) : stk[l][lane];
            have = true;
        }
    }
    return acc;
}

__device__ __forceinline__ void add_out(const IdxParams &p, int32_t r, int col, float4 F) {
    float4 *o = reinterpret_cast<float4 *>(p.out + static_cast<int64_t>(r) * p.ld_out + col);
    const float4 a = *o;
    *o = f4add(a, F);
}

// Sub-slot of quarter q of the tile starting at sorted position p0 (tile index t):
// within a 128-position block at most two split-row tiles start, the last tile
// of one row and the first of the next, so the parity bit keeps them apart.
__device__ __forceinline__ int64_t sub_slot(int32_t p0, int32_t t, int q) {
    return (static_cast<int64_t>(p0 >> 7) * 2 + (t == 0 ? 1 : 0)) * 4 + q;
}

// One quarter (32 members) of one tile of a heavy row, from the list K3 built.
// The last quarter of the tile to arrive (an integer ticket) combines the four
// quarters into the tile partial by the top two levels of the tile's tree; the
// last tile of the row to arrive folds the tile partials in ascending order.
__device__ __noinline__ void heavy_unit(const IdxParams &p, int32_t unit, int lane, float4 (*stk)[32]) {
    const int2 ent = p.heavy[unit >> 2];
    const int q = unit & 3;
    const int32_t k = ent.x, t = ent.y;
    const int32_t s0 = p.seg_start[k];
    const int32_t e0 = p.seg_start[k + 1];
    const int32_t p0 = s0 + t * kSegTile;
    const int cnt_tile = min(kSegTile, e0 - p0);
    const int cnt = min(kSub, cnt_tile - q * kSub);
    const int32_t n_tiles = (e0 - s0 + kSegTile - 1) / kSegTile;
    if (cnt > 0) {
        for (int c0 = 0; c0 < p.D; c0 += 128) {
            const int col = c0 + lane * 4;
            const float4 v = window_sum(p, p0 + q * kSub, cnt, col < p.D ? col : -1, lane, stk);
            if (col < p.D) *reinterpret_cast<float4 *>(p.slots + sub_slot(p0, t, q) * p.D + col) = v;
        }
    }
    __threadfence();
    __syncwarp();
    const int64_t tslot = static_cast<int64_t>(p0 >> 7) * 2 + (t == 0 ? 1 : 0);
    int tq = 0;
    if (lane == 0) tq = atomicAdd(&p.tile_tickets[tslot], 1);
    tq = __shfl_sync(0xffffffffu, tq, 0);
    if (tq != 3) return;
    __threadfence();
    for (int c0 = 0; c0 < p.D; c0 += 128) {
        const int col = c0 + lane * 4;
        if (col >= p.D) continue;
        float4 sq[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq)
            if (qq * kSub < cnt_tile)
                sq[qq] = __ldcg(reinterpret_cast<const float4 *>(p.slots + sub_slot(p0, t, qq) * p.D + col));
        float4 a = sq[0];
        if (cnt_tile > 32) a = f4add(a, sq[1]);
        if (cnt_tile > 64) {
            float4 c = sq[2];
            if (cnt_tile > 96) c = f4add(c, sq[3]);
            a = f4add(a, c);
        }
        *reinterpret_cast<float4 *>(p.slots + sub_slot(p0, t, 0) * p.D + col) = a;
    }
    __threadfence();
    __syncwarp();
    int tk = 0;
    if (lane == 0) {
        p.tile_tickets[tslot] = 0;
        tk = atomicAdd(&p.tickets[k], 1);
    }
    tk = __shfl_sync(0xffffffffu, tk, 0);
    if (tk != n_tiles - 1) return;
    __threadfence();
    for (int c0 = 0; c0 < p.D; c0 += 128) {
        const int col = c0 + lane * 4;
        if (col >= p.D) continue;
        float4 F = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t b0 = 0; b0 < n_tiles; b0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (b0 + u < n_tiles)
                    v[u] = __ldcg(reinterpret_cast<const float4 *>(
                        p.slots + sub_slot(s0 + (b0 + u) * kSegTile, b0 + u, 0) * p.D + col));
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (b0 + u < n_tiles) F = (b0 + u == 0) ? v[u] : f4add(F, v[u]);
        }
        add_out(p, k, col, F);
    }
    if (lane == 0) p.tickets[k] = 0;
}

__device__ void row_unit(const IdxParams &p, int32_t r, int lane, float4 (*stk)[32]) {
    const int32_t s = p.seg_start[r];
    const int32_t e = p.seg_start[r + 1];
    const int32_t n = e - s;
    if (n <= 0) return;
    if (p.seg_tile == 1) {  // purely sequential fold in original order
        for (int c0 = 0; c0 < p.D; c0 += 128) {
            const int col = c0 + lane * 4;
            float4 F = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int32_t q0 = 0; q0 < n; q0 += 32) {
                const int32_t mine = (q0 + lane < n) ? p.perm[s + q0 + lane] : 0;
                const int cnt = min(32, n - q0);
#pragma unroll 4
                for (int u = 0; u < cnt; ++u) {
                    const int32_t row = __shfl_sync(0xffffffffu, mine, u);
                    if (col < p.D) {
                        const float4 v = ld_src4(p, row, col);
                        F = (q0 + u == 0) ? v : f4add(F, v);
                    }
                }
            }
            if (col < p.D) add_out(p, r, col, F);
        }
        return;
    }
    const int W = p.seg_tile;
    const int32_t n_tiles = (n + W - 1) / W;
    if (W == kSegTile && n_tiles > kWarpMaxTiles) return;  // split-row units handle it
    for (int c0 = 0; c0 < p.D; c0 += 128) {
        const int col = c0 + lane * 4;
        const int lcol = col < p.D ? col : -1;
        float4 F = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t t = 0; t < n_tiles; ++t) {
            const int cnt = min(W, n - t * W);
            const float4 P = window_sum(p, s + t * W, cnt, lcol, lane, stk);
            F = (t == 0) ? P : f4add(F, P);
        }
        if (col < p.D) add_out(p, r, col, F);
    }
}

// Small widths (2, 4): a tree over 2 or 4 members, per lane, no stack.
__device__ void row_unit_small(const IdxParams &p, int32_t r, int lane) {
    const int32_t s = p.seg_start[r];
    const int32_t e = p.seg_start[r + 1];
    const int32_t n = e - s;
    if (n <= 0) return;
    const int W = p.seg_tile;
    for (int c0 = 0; c0 < p.D; c0 += 128) {
        const int col = c0 + lane * 4;
        float4 F = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t t0 = 0; t0 < n; t0 += W) {
            const int cnt = min(W, n - t0);
            float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0, v2 = v0, v3 = v0;
            if (col < p.D) {
                v0 = ld_src4(p, p.perm[s + t0], col);
                if (cnt > 1) v1 = ld_src4(p, p.perm[s + t0 + 1], col);
                if (cnt > 2) v2 = ld_src4(p, p.perm[s + t0 + 2], col);
                if (cnt > 3) v3 = ld_src4(p, p.perm[s + t0 + 3], col);
                if (cnt > 1) v0 = f4add(v0, v1);
                if (cnt > 3) v2 = f4add(v2, v3);
                if (cnt > 2) v0 = f4add(v0, v2);
                F = (t0 == 0) ? v0 : f4add(F, v0);
            }
        }
        if (col < p.D) add_out(p, r, col, F);
    }
}

__global__ void __launch_bounds__(kThreads, 3) segsum_kernel(const IdxParams p) {
    __shared__ float4 stack[kWarps][kStackLevels][32];
    const int lane = threadIdx.x & 31;
    float4 (*stk)[32] = stack[threadIdx.x >> 5];
    const int64_t wg = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    // the first 4 x (listed heavy tiles) warps also take one quarter of a heavy tile
    const int64_t n_heavy = (p.seg_tile == kSegTile) ? static_cast<int64_t>(p.hdr->pad[3]) * 4 : 0;
    if (wg < n_heavy) heavy_unit(p, static_cast<int32_t>(wg), lane, stk);
    const int64_t r = wg;
    if (r > p.R) return;
    if (p.seg_tile == 2 || p.seg_tile == 4) row_unit_small(p, static_cast<int32_t>(r), lane);
    else row_unit(p, static_cast<int32_t>(r), lane, stk);
}

struct IdxLayout {
    int32_t nb, n_buckets, n_pblk, max_heavy;
    size_t keys_a, vals_a, perm, skey, hist, offs, bucket_start, seg_start, tickets, tile_tickets, slots;
    size_t bucket_negmin, bucket_max, bucket_key, heavy, total;
};

IdxLayout idx_layout(int64_t N, int64_t R, int64_t D) {
    IdxLayout L{};
    L.nb = static_cast<int32_t>((N + kBlockElems - 1) / kBlockElems);
    L.n_buckets = static_cast<int32_t>((R + 1 + 255) / 256);
    L.n_pblk = static_cast<int32_t>((N + 127) / 128);
    // tiles of rows with more than 8 tiles: at most N/128 plus one ragged tile per such row
    L.max_heavy = static_cast<int32_t>(N / kSegTile + N / (kWarpMaxTiles * kSegTile + 1) + 1);
    size_t o = sizeof(WsHeader);
    auto take = [&](size_t bytes) {
        size_t at = o;
        o += align_up(bytes);
        return at;
    };
    L.keys_a = take(N * 4);
    L.vals_a = take(N * 4);
    L.perm = take(N * 4);
    L.skey = take(N * 4);
    L.hist = take(static_cast<size_t>(kDigits) * L.nb * 4);
    L.offs = take(static_cast<size_t>(kDigits) * L.nb * 4);
    L.bucket_start = take((kDigits + 1) * 4);
    L.seg_start = take((R + 2) * 4);
    L.tickets = take((R + 1) * 4);
    L.tile_tickets = take(static_cast<size_t>(L.n_pblk) * 2 * 4);
    L.slots = take(static_cast<size_t>(L.n_pblk) * 8 * D * 4);
    L.bucket_negmin = take(kDigits * 4);
    L.bucket_max = take(kDigits * 4);
    L.bucket_key = take(kDigits * 4);
    L.heavy = take(static_cast<size_t>(L.max_heavy) * 8);
    L.total = o;
    return L;
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" size_t dgr_index_add_workspace_bytes(int64_t N, int64_t R, int64_t D) {
    if (N < 0 || R < 0 || D < 0 || R + 1 > 65536 || N > INT32_MAX || D > 4096) return 0;
    return idx_layout(N, R, D).total;
}

extern "C" dgr_status dgr_det_index_add(float *out, int64_t R, int64_t D, int64_t ld_out, const float *src,
                                        int64_t ld_src, const int32_t *idx, int64_t N, int32_t seg_tile,
                                        int32_t *bad_count, void *ws, size_t ws_bytes, void *stream) {
    if (R < 0 || D < 0 || N < 0) return DGR_ERR_INVALID_ARG;
    if (!is_pow2(seg_tile) || seg_tile > kSegTile) return DGR_ERR_INVALID_ARG;
    if (R + 1 > 65536 || N > INT32_MAX || D > 4096) return DGR_ERR_UNSUPPORTED;
    if (!out || (N > 0 && (!src || !idx))) return DGR_ERR_INVALID_ARG;
    if (ld_out < D || (N > 0 && ld_src < D)) return DGR_ERR_INVALID_ARG;
    if ((D % 4) != 0 || (ld_out % 4) != 0 || (ld_src % 4) != 0 || !aligned(out, 16) ||
        (src && !aligned(src, 16)) || (idx && !aligned(idx, 4)) || (bad_count && !aligned(bad_count, 4)))
        return DGR_ERR_MISALIGNED;
    const IdxLayout L = idx_layout(N, R, D);
    if (N > 0) {
        if (!ws) return DGR_ERR_INVALID_ARG;
        if (ws_bytes < L.total) return DGR_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(ws, kAlign)) return DGR_ERR_MISALIGNED;
    }
    const size_t ext_out = static_cast<size_t>((R * ld_out + D) * 4);
    const size_t ext_src = N > 0 ? static_cast<size_t>(((N - 1) * ld_src + D) * 4) : 0;
    if (ranges_overlap(out, ext_out, src, ext_src) || ranges_overlap(out, ext_out, idx, N * 4) ||
        ranges_overlap(out, ext_out, bad_count, bad_count ? 4 : 0) ||
        (N > 0 && ranges_overlap(out, ext_out, ws, L.total)))
        return DGR_ERR_ALIAS;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        if (bad_count && cudaMemsetAsync(bad_count, 0, 4, s) != cudaSuccess) return DGR_ERR_CUDA;
        return DGR_OK;
    }
    IdxParams p{};
    p.idx = idx;
    p.N = static_cast<int32_t>(N);
    p.R = static_cast<int32_t>(R);
    p.D = static_cast<int32_t>(D);
    p.nb = L.nb;
    p.n_buckets = L.n_buckets;
    p.n_pblk = L.n_pblk;
    p.seg_tile = seg_tile;
    p.src = src;
    p.ld_src = ld_src;
    p.out = out;
    p.ld_out = ld_out;
    p.bad_count = bad_count;
    char *w = static_cast<char *>(ws);
    p.hdr = reinterpret_cast<WsHeader *>(w);
    p.keys_a = reinterpret_cast<int32_t *>(w + L.keys_a);
    p.vals_a = reinterpret_cast<int32_t *>(w + L.vals_a);
    p.perm = reinterpret_cast<int32_t *>(w + L.perm);
    p.skey = reinterpret_cast<int32_t *>(w + L.skey);
    p.hist = reinterpret_cast<int32_t *>(w + L.hist);
    p.offs = reinterpret_cast<int32_t *>(w + L.offs);
    p.bucket_start = reinterpret_cast<int32_t *>(w + L.bucket_start);
    p.seg_start = reinterpret_cast<int32_t *>(w + L.seg_start);
    p.tickets = reinterpret_cast<int32_t *>(w + L.tickets);
    p.tile_tickets = reinterpret_cast<int32_t *>(w + L.tile_tickets);
    p.slots = reinterpret_cast<float *>(w + L.slots);
    p.bucket_negmin = reinterpret_cast<int32_t *>(w + L.bucket_negmin);
    p.bucket_max = reinterpret_cast<int32_t *>(w + L.bucket_max);
    p.bucket_key = reinterpret_cast<int32_t *>(w + L.bucket_key);
    p.heavy = reinterpret_cast<int2 *>(w + L.heavy);
    count_kernel<<<L.nb, kThreads, 0, s>>>(p);
    scatter_high_kernel<<<L.nb, kThreads, 0, s>>>(p);
    bucket_kernel<<<L.n_buckets, kThreads, 0, s>>>(p);
    if (D > 0) {
        const int64_t heavy_warps = seg_tile == kSegTile ? static_cast<int64_t>(L.max_heavy) * 4 : 0;
        const int64_t warps = (R + 1) > heavy_warps ? (R + 1) : heavy_warps;
        const int64_t grid = (warps + kWarps - 1) / kWarps;
        if (grid > INT32_MAX) return DGR_ERR_UNSUPPORTED;
        segsum_kernel<<<static_cast<unsigned>(grid), kThreads, 0, s>>>(p);
    }
    return launch_status();
}
