// Deterministic index_add: stable radix sort by destination, then segmented
// pairwise sums in original order, padding routed to the dummy row R.
//
// Megatron-LM PR #7441 (DSv4 --deterministic-mode), Source 3: the atomic-free
// dK is an index_add done as a stable sort plus a (prefix) sum, with padding
// slots spread over dummy rows that the caller drops. Four launches:
//   hist     - map idx to keys (idx outside [0, R) -> R; outside [-1, R) is
//              counted); each 2048-element tile stores its low-byte digit
//              counts and adds its low- and high-byte histograms and its
//              per-key counts to the global ones (integer atomics; the
//              padding key R summed in the block first).
//   pass 0/1 - stable LSD radix passes by the low, then the high byte. Each
//              tile ranks its elements in original order with warp
//              match/ballot and per-warp digit counters; a digit's offset is
//              its global base plus the earlier tiles' counts of it, summed
//              32 tiles at a time back to the nearest tile that has already
//              published its inclusive count. Every count is there before the
//              pass starts (pass 0 adds, per element, to the digit counts of
//              the pass-1 tile it lands in), so nothing waits. Pass 1 writes
//              the sorted keys and the permutation. Its first tiles also
//              turn the per-key counts into seg_start[], one 256-key bucket
//              each (the bucket's base from the high-byte histogram plus a
//              scan of its keys' counts), and list rows longer than 32 tiles.
//   segsum   - persistent warps, each an equal share of the sorted order: the
//              rows starting in the share as one stream of 8-member groups,
//              summed by the pairwise tree over tiles of 128 members and
//              folded tile by tile, then out[r] += sum with one rounding. A
//              row longer than one tile is split by tile; the tile partials
//              go to slots and are folded in order by the warp completing the
//              last tile (an integer ticket) or, for rows longer than 32
//              tiles, by a fold block.
// Every scratch word a launch leaves non-zero is cleared by a later launch of
// the same call (segsum clears the sort's counters, even with no columns), so
// a workspace zeroed once serves every call.
// Integer atomics only count or hand out tile numbers; no floating-point
// value depends on timing.
#include "dgr_common.cuh"

namespace dgr {
namespace {

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortItems = 8;
constexpr int kSortTile = kSortThreads * kSortItems;  // 2048 elements per sort tile
constexpr int kDigits = 256;
constexpr int kSegTile = 128;
constexpr int kSplitMin = kSegTile;    // rows longer than one tile are split by tile
constexpr int kWarpFoldTiles = 32;     // split rows up to 32 tiles: folded by one warp
constexpr int kMaxFoldBlocks = 16;     // longer rows: folded by up to 16 fold blocks

struct IdxParams {
    const int32_t *idx;
    int32_t N, R, D;
    int32_t nb;         // sort tiles
    int32_t n_buckets;  // 256-key buckets of the keys 0..R (segment starts, one pass-1 block each)
    int32_t n_pblk;  // 128-position blocks of the sorted order (slot indexing)
    int32_t seg_tile;
    const float *src;
    int64_t ld_src;
    float *out;
    int64_t ld_out;
    int32_t *bad_count;
    int32_t *keys_a, *vals_a, *perm, *skey, *seg_start, *tickets;
    int32_t *hist;               // [2][256] global digit histograms (low byte, high byte)
    int32_t *count;              // [R + 1] elements per key
    int32_t *cnt;                // [2][nb][256] per-tile digit counts of the two passes
    int32_t *incl;               // [2][nb][256] published inclusive counts (bit 31: published)
    int32_t *heavy_rows;         // split rows longer than kWarpFoldTiles tiles (fold-block work)
    int32_t max_fold_rows;       // capacity of heavy_rows
    Sched sched_tiles;           // which block takes which sort tile (hist, pass 0)
    Sched sched_pass1;           // the same over pass 1's items (sort tiles and key buckets)
    Sched sched_warps;           // segsum: the setting, bound on the device to its warp count
    float *slots;
    WsHeader *hdr;  // pad[2]: bad-index total, pad[3]: fold-row count, pad[8..10]: layout tag
};

// Layout tag (header words 8-10): N, R + 1 and a constant, all non-zero,
// written by hist's block 0 on the first call on a zeroed workspace. The
// regions of the workspace move with N and R, and the arrays one call leaves
// behind (keys, permutation) would be read as counters by a call of other
// sizes, so every launch of a call checks the tag before it writes anything.
// A word is accepted when it is still zero (a fresh workspace whose tag hist
// is writing) or holds this call's value; any other value is a workspace of
// other sizes, which nobody rewrites, so every launch can read the tag early,
// before its dependency wait, and all of them reach the same answer.
constexpr int32_t kTagMagic = 0x31584449;
constexpr int kTagWord = 8;

__device__ __forceinline__ bool tag_word_ok(int32_t have, int32_t want) { return have == 0 || have == want; }

__device__ __forceinline__ bool tag_ok(const IdxParams &p) {
    const volatile int32_t *t = p.hdr->pad + kTagWord;
    const int32_t t0 = t[0], t1 = t[1], t2 = t[2];
    return tag_word_ok(t0, p.N) && tag_word_ok(t1, p.R + 1) && tag_word_ok(t2, kTagMagic);
}

__device__ __forceinline__ int32_t clampi(int32_t v, int32_t lo, int32_t hi) { return min(max(v, lo), hi); }

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

// Programmatic dependent launch: the next launch of the call may start its
// blocks early (launch_dependents); a launch reads what the previous one
// wrote only after grid_dep_wait, which returns once that launch has
// completed and its writes are visible.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// hist: global digit histograms of the two passes, and the bad-index count.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSortThreads) hist_kernel(const IdxParams p) {
    __shared__ int32_t h[2][kDigits];
    __shared__ int32_t bad_block, pad_block, tag_good;
    const int tid = threadIdx.x;
    launch_dependents();
    // sort tiles in the schedule's order; with a capped grid a block takes several
    int32_t it = blockIdx.x;
    int32_t tile = static_cast<int32_t>(sched_item(p.sched_tiles, static_cast<uint32_t>(it)));
    int32_t v[kSortItems];
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
        const int64_t e = static_cast<int64_t>(tile) * kSortTile + r * kSortThreads + tid;
        v[r] = 0;
        ldg_nc_b32_if(v[r], p.idx + e, e < p.N);
    }
    if (tid == 0) {
        tag_good = tag_ok(p);
        if (blockIdx.x == 0) {
            if (tag_good) {
                p.hdr->pad[3] = 0;  // fold-row list of this call starts empty
                p.hdr->pad[kTagWord] = p.N;
                p.hdr->pad[kTagWord + 1] = p.R + 1;
                p.hdr->pad[kTagWord + 2] = kTagMagic;
            } else {
                record_error(p.hdr, DGR_ERR_INVALID_ARG, 40);
            }
        }
    }
    for (;;) {
        h[0][tid] = 0;
        h[1][tid] = 0;
        if (tid == 0) {
            bad_block = 0;
            pad_block = 0;
        }
        __syncthreads();
        if (!tag_good) return;  // a workspace laid out for other sizes: nothing is written
        int my_bad = 0;
#pragma unroll
        for (int r = 0; r < kSortItems; ++r) {
            const int64_t e = static_cast<int64_t>(tile) * kSortTile + r * kSortThreads + tid;
            if (e >= p.N) continue;
            bool bad = false;
            const int32_t k = map_key(v[r], p.R, bad);
            my_bad += bad ? 1 : 0;
            atomicAdd(&h[0][k & 255], 1);
            atomicAdd(&h[1][k >> 8], 1);
            if (k == p.R) atomicAdd(&pad_block, 1);
            else atomicAdd(&p.count[k], 1);
        }
        if (my_bad) atomicAdd(&bad_block, my_bad);
        __syncthreads();
        if (tid == 0 && pad_block) atomicAdd(&p.count[p.R], pad_block);
        p.cnt[static_cast<int64_t>(tile) * kDigits + tid] = h[0][tid];
        if (h[0][tid]) atomicAdd(&p.hist[tid], h[0][tid]);
        if (h[1][tid]) atomicAdd(&p.hist[kDigits + tid], h[1][tid]);
        if (tid == 0 && bad_block) atomicAdd(&p.hdr->pad[2], bad_block);
        it += gridDim.x;
        if (it >= p.nb) return;
        tile = static_cast<int32_t>(sched_item(p.sched_tiles, static_cast<uint32_t>(it)));
        __syncthreads();  // the block's counts of the last tile are read: reuse the arrays
#pragma unroll
        for (int r = 0; r < kSortItems; ++r) {
            const int64_t e = static_cast<int64_t>(tile) * kSortTile + r * kSortThreads + tid;
            v[r] = 0;
            ldg_nc_b32_if(v[r], p.idx + e, e < p.N);
        }
    }
}

// Stable in-warp ranking: warp w owns its elements in rounds of 32
// (round-major, lane order = element order). Returns each element's rank
// among equal digits inside its warp; cnt[w][d] ends as the warp's digit
// counts.
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
// pass 0/1: stable radix pass by the low (0) or high (1) byte of the key.
// ---------------------------------------------------------------------------
template <int PASS>
__device__ __forceinline__ int pass_digit(int32_t key) {
    return PASS == 0 ? (key & 255) : (key >> 8);
}

constexpr int kLookWindow = 32;
constexpr int32_t kPublished = static_cast<int32_t>(0x80000000u);

// Relaxed 32-bit load under a predicate; v keeps its value otherwise.
__device__ __forceinline__ void ld_relaxed_b32_if(int32_t &v, const int32_t *a, bool pred) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q ld.relaxed.gpu.global.b32 %0, [%1];\n\t}"
        : "+r"(v)
        : "l"(a), "r"(static_cast<int>(pred))
        : "memory");
}

// Count of digit d in the tiles before tile b: the earlier tiles' counts,
// nearest first, kLookWindow at a time, until a tile whose inclusive count is
// already published (it then replaces the rest); then tile b publishes its
// own inclusive count. The counts come from earlier launches, so nothing
// waits; an inclusive word holds all it publishes, so relaxed accesses
// suffice. The first window is loaded early (look_load) and consumed late
// (look_finish), with the tile's ranking in between.
struct LookWin {
    int32_t c[kLookWindow], f[kLookWindow];
};

__device__ __forceinline__ void look_load(LookWin &L, const int32_t *cnt, const int32_t *incl, int32_t j_hi, int d) {
#pragma unroll
    for (int u = 0; u < kLookWindow; ++u) {
        const int64_t at = static_cast<int64_t>(j_hi - u) * kDigits + d;
        L.c[u] = 0;
        L.f[u] = 0;
        ld_relaxed_b32_if(L.f[u], incl + at, j_hi - u >= 0);
        ldg_nc_b32_if(L.c[u], cnt + at, j_hi - u >= 0);
    }
}

__device__ __forceinline__ int32_t look_finish(LookWin &L, const int32_t *cnt, int32_t *incl, int32_t b, int d,
                                               int32_t count) {
    int32_t excl = 0;
    for (int32_t j_hi = b - 1; j_hi >= 0; j_hi -= kLookWindow) {
        if (j_hi != b - 1) look_load(L, cnt, incl, j_hi, d);
        bool done = false;
#pragma unroll
        for (int u = 0; u < kLookWindow; ++u) {
            if (done) continue;
            if (L.f[u] & kPublished) {
                excl += L.f[u] & ~kPublished;
                done = true;
            } else {
                excl += L.c[u];
            }
        }
        if (done) break;
    }
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(incl + static_cast<int64_t>(b) * kDigits + d),
                 "r"(kPublished | (excl + count))
                 : "memory");
    return excl;
}

// Sum over tiles [0, b) of the digit counts, by 8 warps: warp v takes tiles
// v, v + 8, ..., lane l digits 8l .. 8l + 7 (two 16-byte loads a tile), 8
// tiles a lane in flight; the 8 partial sums go to red[v][].
__device__ __forceinline__ void direct_prefix(const int32_t *cnt, int32_t b, int v, int lane, int32_t (*red)[kDigits]) {
    int32_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int32_t j0 = v; j0 < b; j0 += 8 * kSortWarps) {
        uint4 x[16];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t j = j0 + u * kSortWarps;
            x[2 * u] = x[2 * u + 1] = make_uint4(0u, 0u, 0u, 0u);
            ldg_nc_v4u_if(x[2 * u], cnt + static_cast<int64_t>(j) * kDigits + lane * 8, j < b);
            ldg_nc_v4u_if(x[2 * u + 1], cnt + static_cast<int64_t>(j) * kDigits + lane * 8 + 4, j < b);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            acc[(u & 1) * 4 + 0] += static_cast<int32_t>(x[u].x);
            acc[(u & 1) * 4 + 1] += static_cast<int32_t>(x[u].y);
            acc[(u & 1) * 4 + 2] += static_cast<int32_t>(x[u].z);
            acc[(u & 1) * 4 + 3] += static_cast<int32_t>(x[u].w);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[v][lane * 8 + i] = acc[i];
}

constexpr int kPassThreads = 2 * kSortThreads;  // 8 ranking warps, 8 prefix warps
constexpr int32_t kDirectTiles = 512;           // tiles below this sum the earlier counts directly

template <int PASS>
__global__ void __launch_bounds__(kPassThreads) pass_kernel(const IdxParams p) {
    __shared__ int32_t cnt[kSortWarps][kDigits];
    __shared__ int32_t red[kSortWarps][kDigits];
    __shared__ int32_t gbase[kDigits];    // global position of this tile's first element of each digit
    __shared__ int32_t lbase[kDigits];    // local position of the same
    __shared__ int32_t excl_s[kDigits];
    __shared__ int32_t dbase_s[kDigits];  // global position of each digit's first element
    __shared__ int32_t wsum[kSortWarps];
    __shared__ int32_t lsum[kSortWarps];
    __shared__ int32_t csum[kSortWarps];
    __shared__ int32_t sk[kSortTile], sv[kSortTile];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int64_t tiles = static_cast<int64_t>(p.nb) * kDigits;
    const int32_t *cnt_g = p.cnt + PASS * tiles;
    int32_t *incl_g = p.incl + PASS * tiles;
    // items: sort tiles, and in pass 1 also key buckets where there are more
    // buckets than tiles; handed out in the schedule's order (with a capped
    // grid a block takes several). No item waits for another.
    const int32_t n_items = PASS == 0 ? p.nb : max(p.nb, p.n_buckets);
    const Sched &sc = PASS == 0 ? p.sched_tiles : p.sched_pass1;
    __shared__ int32_t s_good;
    for (int q = tid; q < kSortWarps * kDigits; q += kPassThreads) (&cnt[0][0])[q] = 0;
    launch_dependents();
    if (tid == 0) s_good = tag_ok(p);  // read while the previous launch finishes
    grid_dep_wait();
    __syncthreads();
    if (!s_good) return;  // hist refused the workspace
    for (int32_t it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int32_t b = static_cast<int32_t>(sched_item(sc, static_cast<uint32_t>(it)));
        // pass 1's first n_buckets items also own the segment starts of bucket b
        const bool seg_owner = PASS == 1 && b < p.n_buckets;
        const bool sort_tile = b < p.nb;  // pass 1 may have more items than tiles (more buckets)
        if (it != static_cast<int32_t>(blockIdx.x)) {
            for (int q = tid; q < kSortWarps * kDigits; q += kPassThreads) (&cnt[0][0])[q] = 0;
            __syncthreads();
        }
        int32_t key[kSortItems], val[kSortItems], rank[kSortItems];
        int32_t gx = 0, my_count = 0;
        int32_t kc = 0, kx = 0;  // prefix warps of a segment-start owner: the key's count, warp prefix
        if (w < kSortWarps) {
            // ranking warps: warp w owns elements [b*2048 + w*256, +256) in 8 rounds of 32
            const int64_t e0 = static_cast<int64_t>(b) * kSortTile + w * (kSortItems * 32) + lane;
#pragma unroll
            for (int r = 0; r < kSortItems; ++r) {
                const int64_t e = e0 + r * 32;
                key[r] = 0;
                val[r] = static_cast<int32_t>(e);
                if (PASS == 0) {
                    ldg_nc_b32_if(key[r], p.idx + e, e < p.N);
                } else {
                    ldg_nc_b32_if(key[r], p.keys_a + e, e < p.N);
                    ldg_nc_b32_if(val[r], p.vals_a + e, e < p.N);
                }
            }
            const int32_t hc = __ldcg(&p.hist[PASS * kDigits + tid]);
            if (sort_tile) my_count = __ldcg(&cnt_g[static_cast<int64_t>(b) * kDigits + tid]);
#pragma unroll
            for (int r = 0; r < kSortItems; ++r) {
                const int64_t e = e0 + r * 32;
                if (e >= p.N) {
                    key[r] = -1;
                } else if (PASS == 0) {
                    bool bad = false;
                    key[r] = map_key(key[r], p.R, bad);
                } else {
                    key[r] = clampi(key[r], 0, p.R);  // a key read back from the workspace stays a key
                }
            }
#pragma unroll
            for (int r = 0; r < kSortItems; ++r)
                warp_rank(key[r] >= 0 ? pass_digit<PASS>(key[r]) : 0, key[r] >= 0, cnt, w, rank[r]);
            // exclusive scans over digits of the global histogram (global digit
            // bases) and of this tile's counts (local digit bases)
            int32_t gi = hc, li = my_count;
#pragma unroll
            for (int s = 1; s < 32; s <<= 1) {
                const int32_t tg = __shfl_up_sync(0xffffffffu, gi, s);
                const int32_t tl = __shfl_up_sync(0xffffffffu, li, s);
                if (lane >= s) {
                    gi += tg;
                    li += tl;
                }
            }
            if (lane == 31) {
                wsum[w] = gi;
                lsum[w] = li;
            }
            gx = gi - hc;
            lbase[tid] = li - my_count;
        } else {
            if (seg_owner) {  // the counts of keys 256b .. 256b + 255, scanned within each warp
                const int32_t k = b * kDigits + (tid - kSortThreads);
                if (k <= p.R) kc = __ldcg(&p.count[k]);
                int32_t ci = kc;
#pragma unroll
                for (int s = 1; s < 32; s <<= 1) {
                    const int32_t tv = __shfl_up_sync(0xffffffffu, ci, s);
                    if (lane >= s) ci += tv;
                }
                if (lane == 31) csum[w - kSortWarps] = ci;
                kx = ci - kc;
            }
            if (sort_tile && b < kDirectTiles) direct_prefix(cnt_g, b, w - kSortWarps, lane, red);
        }
        __syncthreads();
        if (w < kSortWarps) {
            int32_t lx = lbase[tid];
            for (int ww = 0; ww < w; ++ww) {
                gx += wsum[ww];
                lx += lsum[ww];
            }
            lbase[tid] = lx;
            dbase_s[tid] = gx;
            int32_t run = 0;
#pragma unroll
            for (int ww = 0; ww < kSortWarps; ++ww) {
                const int32_t c = cnt[ww][tid];
                cnt[ww][tid] = run;
                run += c;
            }
        } else {
            const int d = tid - kSortThreads;
            const int32_t mine = sort_tile ? __ldcg(&cnt_g[static_cast<int64_t>(b) * kDigits + d]) : 0;
            int32_t excl = 0;
            if (!sort_tile) {
            } else if (b < kDirectTiles) {
#pragma unroll
                for (int v = 0; v < kSortWarps; ++v) excl += red[v][d];
                asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(incl_g + static_cast<int64_t>(b) * kDigits + d),
                             "r"(kPublished | (excl + mine))
                             : "memory");
            } else {
                LookWin L;
                look_load(L, cnt_g, incl_g, b - 1, d);
                excl = look_finish(L, cnt_g, incl_g, b, d, mine);
            }
            excl_s[d] = excl;
            if (seg_owner)
                for (int ww = 0; ww < w - kSortWarps; ++ww) kx += csum[ww];
        }
        __syncthreads();
        if (w < kSortWarps) {
            gbase[tid] = gx + excl_s[tid];
            // the tile in digit order in shared memory
#pragma unroll
            for (int r = 0; r < kSortItems; ++r) {
                if (key[r] < 0) continue;
                const int d = pass_digit<PASS>(key[r]);
                // the local bases come from counts in the workspace: keep the
                // position inside the tile whatever they hold
                const int32_t lp = clampi(lbase[d] + cnt[w][d] + rank[r], 0, kSortTile - 1);
                sk[lp] = key[r];
                sv[lp] = val[r];
            }
        } else if (seg_owner) {
            // segment starts of bucket b: the bucket's first position plus the
            // counts of its smaller keys; its long rows go on the fold-block list
            // (in any order: each row is folded by one block, the same way)
            const int32_t k = b * kDigits + (tid - kSortThreads);
            if (k <= p.R) {
                p.seg_start[k] = clampi(dbase_s[b] + kx, 0, p.N);
                if (k == p.R) p.seg_start[p.R + 1] = p.N;
                if (p.seg_tile == kSegTile && kc > kWarpFoldTiles * kSegTile) {
                    const int32_t at = atomicAdd(&p.hdr->pad[3], 1);
                    if (at < p.max_fold_rows) p.heavy_rows[at] = k;
                }
                p.count[k] = 0;  // read no more: cleared for the next call
            }
            if (b == 0 && tid == kSortThreads) {  // every hist block has counted by now
                const int32_t bad = atomicAdd(&p.hdr->pad[2], 0);
                if (p.bad_count) *p.bad_count = bad;
                p.hdr->pad[2] = 0;
            }
        }
        __syncthreads();
        // each digit's run written out contiguously
        const int n_here = static_cast<int>(
            min(static_cast<int64_t>(kSortTile), static_cast<int64_t>(p.N) - static_cast<int64_t>(b) * kSortTile));
#pragma unroll
        for (int r = 0; r < kSortTile / kPassThreads; ++r) {
            const int i = r * kPassThreads + tid;
            if (i >= n_here) continue;
            const int32_t k = clampi(sk[i], 0, p.R);
            const int d = pass_digit<PASS>(k);
            // digit bases come from counts in the workspace: the write stays in [0, N)
            const int32_t pos = clampi(gbase[d] + (i - lbase[d]), 0, p.N - 1);
            if (PASS == 0) {
                p.keys_a[pos] = k;
                p.vals_a[pos] = sv[i];
                atomicAdd(&p.cnt[tiles + static_cast<int64_t>(pos / kSortTile) * kDigits + (k >> 8)], 1);
            } else {
                p.perm[pos] = sv[i];
                p.skey[pos] = k;
            }
        }
        // pass 0's inclusive words are read no more: clear them for the next call
        if (PASS == 1 && sort_tile && tid < kDigits) p.incl[static_cast<int64_t>(b) * kDigits + tid] = 0;
        __syncthreads();  // the item's shared arrays are read: the next item may reuse them
    }
}

// ---------------------------------------------------------------------------
// segsum: segmented sums.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float4 f4add(float4 a, float4 b) {
    // two packed adds, the same bits as four scalar ones
    const float2 lo = add2(make_float2(a.x, a.y), make_float2(b.x, b.y));
    const float2 hi = add2(make_float2(a.z, a.w), make_float2(b.z, b.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ void add_out(const IdxParams &p, int32_t r, int col, float4 F) {
    float4 *o = reinterpret_cast<float4 *>(p.out + static_cast<int64_t>(r) * p.ld_out + col);
    const float4 a = *o;
    *o = f4add(a, F);
}

// Slot of the partial of the split-row tile starting at sorted position p0:
// within a 128-position block at most two split-row tiles start, the last
// tile of one row and the first tile (tfirst) of the next, so the parity bit
// keeps them apart.
__device__ __forceinline__ float4 *tile_slot(const IdxParams &p, int64_t p0, bool tfirst, int col) {
    return reinterpret_cast<float4 *>(p.slots + ((p0 >> 7) * 2 + (tfirst ? 1 : 0)) * p.D + col);
}

// Ordered fold of the tile partials of a split row of at most kWarpFoldTiles
// tiles by one warp, then out[k] += F.
__device__ void warp_fold(const IdxParams &p, int32_t k, int64_t s0, int32_t n_tiles, int lane) {
    for (int c0 = 0; c0 < p.D; c0 += 128) {
        const int col = c0 + lane * 4;
        if (col >= p.D) continue;
        float4 F = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t b0 = 0; b0 < n_tiles; b0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                ldcg_v4f_if(v[u], tile_slot(p, s0 + static_cast<int64_t>(b0 + u) * kSegTile, b0 + u == 0, col),
                            b0 + u < n_tiles);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (b0 + u < n_tiles) F = (b0 + u == 0) ? v[u] : f4add(F, v[u]);
        }
        add_out(p, k, col, F);
    }
}

// A split-row tile is done for one column block: its partial goes to its slot
// and the row counts it (an integer ticket). The last of the row's
// tiles x column blocks to arrive folds a row of at most kWarpFoldTiles tiles;
// a longer row is folded by a fold block.
// (long_by_warp: no fold block runs - a one-block grid - so the last tile
// folds a longer row too.)
__device__ __noinline__ void tile_done(const IdxParams &p, int32_t k, int32_t p0, bool tfirst, float4 P, int col,
                                       bool act, int lane, bool long_by_warp) {
    if (act) *tile_slot(p, p0, tfirst, col) = P;
    __threadfence();
    __syncwarp();
    int32_t s0 = 0, e0 = 0, tk = 0;
    if (lane == 0) {
        s0 = clampi(p.seg_start[k], 0, p.N);
        e0 = clampi(p.seg_start[k + 1], s0, p.N);
        tk = atomicAdd(&p.tickets[k], 1);
    }
    s0 = __shfl_sync(0xffffffffu, s0, 0);
    e0 = __shfl_sync(0xffffffffu, e0, 0);
    tk = __shfl_sync(0xffffffffu, tk, 0);
    const int32_t n_tiles = (e0 - s0 + kSegTile - 1) / kSegTile;
    const int32_t n_cb = (p.D + 127) / 128;
    if ((n_tiles > kWarpFoldTiles && !long_by_warp) || tk != n_tiles * n_cb - 1) return;
    __threadfence();
    warp_fold(p, k, s0, n_tiles, lane);
    if (lane == 0) p.tickets[k] = 0;
}

// Work of 32 consecutive keys, one per lane, cut into groups of gs members
// (gs = 8, or the tile width when it is smaller) aligned to the row start.
// The warp takes an unsplit row whole if it starts in its share [P0, P1), and
// of a split row the tiles whose first member lies there.
struct KeyRows {
    int32_t st, L, G, inc;  // first member taken, members taken, groups, inclusive prefix of G
    int32_t ga0, sp;        // group index (within the row) of the first group taken; split row
    int32_t kc, T;          // first key, total groups (uniform)
};

__device__ __forceinline__ void load_seg(const IdxParams &p, int32_t kc, int32_t k_end, int lane, int32_t &st,
                                         int32_t &en) {
    const int32_t k = kc + lane;
    st = en = 0;
    ldg_nc_b32_if(st, &p.seg_start[k], lane < k_end - kc);
    ldg_nc_b32_if(en, &p.seg_start[k + 1], lane < k_end - kc);
    // segment starts are workspace words: every row stays inside [0, N)
    st = clampi(st, 0, p.N);
    en = clampi(en, st, p.N);
}

__device__ __forceinline__ KeyRows key_rows(int32_t kc, int32_t k_end, int32_t st, int32_t en, int gs, bool split_on,
                                            int32_t P0, int32_t P1, int lane) {
    KeyRows R;
    R.kc = kc;
    const bool in = lane < k_end - kc;
    const int32_t L = en - st;
    R.sp = (split_on && L > kSplitMin) ? 1 : 0;
    R.st = st;
    R.L = (st >= P0 && st < P1) ? L : 0;  // an unsplit row is the warp's if it starts in [P0, P1)
    R.ga0 = 0;
    if (R.sp) {
        const int32_t n_t = (L + kSegTile - 1) / kSegTile;
        const int32_t t_lo = st >= P0 ? 0 : (P0 - st + kSegTile - 1) / kSegTile;
        const int32_t t_hi = min(n_t, static_cast<int32_t>((static_cast<int64_t>(P1) - st + kSegTile - 1) / kSegTile));
        if (t_hi <= t_lo) {
            R.L = 0;
        } else {
            const int64_t a = static_cast<int64_t>(st) + static_cast<int64_t>(t_lo) * kSegTile;
            const int64_t b = min(static_cast<int64_t>(en), static_cast<int64_t>(st) + static_cast<int64_t>(t_hi) * kSegTile);
            R.st = static_cast<int32_t>(a);
            R.L = static_cast<int32_t>(b - a);
            R.ga0 = t_lo * (kSegTile / 8);
        }
    }
    R.G = (in && R.L > 0) ? (R.L + gs - 1) / gs : 0;
    int32_t inc = R.G;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += t;
    }
    R.inc = inc;
    R.T = __shfl_sync(0xffffffffu, inc, 31);
    return R;
}

// A group's descriptor in one word: members (bits 0-3), first group (bit 4:
// of its row, or of its tile in a split row), last group (bit 5: of its row,
// or of its tile in a split row), index in its tile (bits 6-9), split row
// (bit 10), group of the row's first tile (bit 11), row key (bits 12-28).
__device__ __forceinline__ int32_t pack_group(int32_t key, int nv, bool first, bool last, int gi, bool sp, bool tfirst) {
    return nv | (first << 4) | (last << 5) | (gi << 6) | (sp << 10) | (tfirst << 11) | (key << 12);
}
__device__ __forceinline__ int gd_nv(int32_t d) { return d & 15; }
__device__ __forceinline__ bool gd_first(int32_t d) { return (d >> 4) & 1; }
__device__ __forceinline__ bool gd_last(int32_t d) { return (d >> 5) & 1; }
__device__ __forceinline__ int gd_gi(int32_t d) { return (d >> 6) & 15; }
__device__ __forceinline__ bool gd_split(int32_t d) { return (d >> 10) & 1; }
__device__ __forceinline__ bool gd_tfirst(int32_t d) { return (d >> 11) & 1; }
__device__ __forceinline__ int32_t gd_key(int32_t d) { return d >> 12; }

// Four consecutive groups: lane l holds member (l & 7) of group q0 + (l >> 3).
struct Quad {
    int32_t pq;    // that member's perm entry
    int32_t desc;  // the group's descriptor
    int32_t aux;   // first sorted position of the group's tile
    int32_t n;     // groups in the quad (uniform)
};

__device__ __forceinline__ Quad make_quad(const IdxParams &p, const KeyRows &R, int32_t q0, int gs, int gpt, int lane) {
    const unsigned full = 0xffffffffu;
    const int32_t q = q0 + (lane >> 3);
    const int u = lane & 7;
    int r = 0;  // rows whose groups end at or before q: q's row
#pragma unroll
    for (int s = 16; s; s >>= 1)
        if (__shfl_sync(full, R.inc, r + s - 1) <= q) r += s;
    const int32_t Gr = __shfl_sync(full, R.G, r), incr = __shfl_sync(full, R.inc, r);
    const int32_t str = __shfl_sync(full, R.st, r), Lr = __shfl_sync(full, R.L, r);
    const int32_t ga0 = __shfl_sync(full, R.ga0, r);
    const bool sp = __shfl_sync(full, R.sp, r) != 0;
    const bool in = q < R.T;
    const int32_t g = q - (incr - Gr);
    const int nv = in ? min(gs, Lr - g * gs) : 0;
    const int32_t ga = ga0 + g;
    const int gi = ga & (gpt - 1);
    const int32_t mpos = str + g * gs;
    Quad Q;
    Q.desc = pack_group(R.kc + r, nv, sp ? gi == 0 : g == 0, g == Gr - 1 || (sp && gi == gpt - 1), gi, sp, ga < gpt);
    Q.aux = mpos - gi * gs;
    Q.pq = 0;
    ldg_nc_b32_if(Q.pq, &p.perm[mpos + u], in && u < nv);
    Q.n = min(4, R.T - q0);
    return Q;
}

// Cursor over the groups of keys [kc, k_end): the current 32 keys' work, the
// next 32 keys' segment starts (prefetched), the next quad to build.
struct GroupCursor {
    KeyRows R;
    int32_t nst, nen, q0, k_end, P0, P1;
};

__device__ __forceinline__ bool next_quad(const IdxParams &p, GroupCursor &c, Quad &Q, int gs, int gpt, bool split_on,
                                          int lane) {
    while (c.q0 >= c.R.T) {
        if (c.k_end - c.R.kc <= 32) return false;
        const int32_t kc = c.R.kc + 32;
        c.R = key_rows(kc, c.k_end, c.nst, c.nen, gs, split_on, c.P0, c.P1, lane);
        if (c.k_end - kc > 32) load_seg(p, kc + 32, c.k_end, lane, c.nst, c.nen);
        c.q0 = 0;
    }
    Q = make_quad(p, c.R, c.q0, gs, gpt, lane);
    c.q0 += 4;
    return true;
}

// A tile's group stack in registers: level l holds the sum of a complete
// block of 2^l groups waiting for its right sibling (at most 16 groups of 8
// in a tile of 128, so five levels).
struct GStack {
    float4 s0, s1, s2, s3, s4;
};

// Group gi of its tile joins the blocks it closes (the pairwise tree, bottom-up).
__device__ __forceinline__ void gpush(GStack &S, int gi, float4 v) {
    if (!(gi & 1)) {
        S.s0 = v;
        return;
    }
    v = f4add(S.s0, v);
    if (!(gi & 2)) {
        S.s1 = v;
        return;
    }
    v = f4add(S.s1, v);
    if (!(gi & 4)) {
        S.s2 = v;
        return;
    }
    v = f4add(S.s2, v);
    if (!(gi & 8)) {
        S.s3 = v;
        return;
    }
    S.s4 = f4add(S.s3, v);
}

// Partial of a tile holding c groups: the complete blocks of the set bits of
// c, smallest first, each larger (earlier) block on the left - the canonical
// tree with the absent leaves past the end passing their sibling up.
__device__ __forceinline__ float4 gpartial(const GStack &S, int c) {
    float4 acc = S.s0;
    bool have = (c & 1) != 0;
    if (c & 2) {
        acc = have ? f4add(S.s1, acc) : S.s1;
        have = true;
    }
    if (c & 4) {
        acc = have ? f4add(S.s2, acc) : S.s2;
        have = true;
    }
    if (c & 8) {
        acc = have ? f4add(S.s3, acc) : S.s3;
        have = true;
    }
    if (c & 16) acc = have ? f4add(S.s4, acc) : S.s4;
    return acc;
}

// 16-byte asynchronous copy global -> shared (L2 only), under a predicate.
__device__ __forceinline__ void cp_async16_if(void *smem, const void *gmem, bool pred) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q cp.async.cg.shared.global [%0], [%1], 16;\n\t}" ::"r"(s),
        "l"(gmem), "r"(static_cast<int>(pred))
        : "memory");
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) { cp_async16_if(smem, gmem, true); }

// The same with an L2 eviction-priority policy (src rows: read once, so
// evict_first keeps them from pushing the workspace and out rows out of L2;
// measured 65 -> 59 us a call with L2 flushed before each).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void cp_async16_hint_if(void *smem, const void *gmem, bool pred, uint64_t pol) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %3;\n\t}" ::"r"(s),
        "l"(gmem), "r"(static_cast<int>(pred)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A warp's ring of kStages slots; a slot holds one group: its 8 source rows
// and, on an unsplit row's first group, the row's out[key] (row 8), 16 bytes
// per lane each; the group's descriptor and tile start sit beside the ring.
constexpr int kStages = 3;
constexpr int kSlotRows = 9;
constexpr int kSlotF4 = kSlotRows * 32;
constexpr int kSegThreads = 512;
constexpr int kSegWarps = kSegThreads / 32;
constexpr int kSegSmemBytes = kSegWarps * (kStages * kSlotF4 * 16 + kStages * 2 * 4);

// Copies of group j of quad Q into a slot. Each lane copies (and later reads)
// only its own 16-byte column slice; the descriptor words (dslot) are written
// by lane 0 and read by all lanes after a warp barrier.
__device__ __forceinline__ void issue_group(const IdxParams &p, float4 *slot, int32_t *dslot, const Quad &Q, int j,
                                            int col, bool act, int lane, uint64_t src_pol) {
    const unsigned full = 0xffffffffu;
    const int32_t gd = __shfl_sync(full, Q.desc, j * 8);
    const int32_t aux = __shfl_sync(full, Q.aux, j * 8);
    __syncwarp();
    if (lane == 0) {
        dslot[0] = gd;
        dslot[1] = aux;
    }
    const int nv = gd_nv(gd);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int32_t row = clampi(__shfl_sync(full, Q.pq, j * 8 + u), 0, p.N - 1);  // a perm entry is a row of src
        cp_async16_hint_if(slot + u * 32 + lane, p.src + static_cast<int64_t>(row) * p.ld_src + col, u < nv && act,
                           src_pol);
    }
    cp_async16_if(slot + 8 * 32 + lane, p.out + static_cast<int64_t>(gd_key(gd)) * p.ld_out + col,
                  gd_first(gd) && !gd_split(gd) && act);
}

struct RowAcc {
    float4 F, o;
    int32_t tix;
};

// Group sum by the tile tree's lowest levels in registers (absent members past
// nv pass their sibling up), then the group joins its tile's group stack; a
// tile's last group yields the tile partial. An unsplit row folds its tile
// partials into F in order and its last group writes out[key] + F; a split
// row's tile partial goes to the tile's slot.
__device__ __forceinline__ void consume_group(const IdxParams &p, const float4 *slot, const int32_t *dslot, RowAcc &ra,
                                              GStack &S, int gs, int gpt, int col, bool act, int lane,
                                              bool long_by_warp) {
    __syncwarp();
    const int32_t gd = dslot[0];
    const int nv = gd_nv(gd);
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = slot[u * 32 + lane];
#pragma unroll
    for (int st = 1; st < 8; st *= 2) {
        if (st < gs) {
#pragma unroll
            for (int r = 0; r + st < 8; r += 2 * st)
                if (r + st < nv) v[r] = f4add(v[r], v[r + st]);
        }
    }
    const bool sp = gd_split(gd);
    if (gd_first(gd) && !sp) {
        ra.o = slot[8 * 32 + lane];
        ra.tix = 0;
    }
    const int gi = gd_gi(gd);
    gpush(S, gi, v[0]);
    const bool last = gd_last(gd);
    if (last || gi == gpt - 1) {
        const float4 P = gpartial(S, gi + 1);
        if (sp) {
            tile_done(p, gd_key(gd), dslot[1], gd_tfirst(gd), P, col, act, lane, long_by_warp);
            return;
        }
        ra.F = (ra.tix == 0) ? P : f4add(ra.F, P);
        ++ra.tix;
    }
    if (last && act)
        *reinterpret_cast<float4 *>(p.out + static_cast<int64_t>(gd_key(gd)) * p.ld_out + col) = f4add(ra.o, ra.F);
}

// Warp's share of the sorted order: positions [P0, P1). The warp sums every
// unsplit row that starts there and every split-row tile that starts there:
// keys [k_first, k_end), walked as one stream of groups. Perm entries come one
// quad (4 groups) ahead; source rows land in the warp's shared-memory ring
// kStages - 1 groups ahead of the sums.
__device__ void walk(const IdxParams &p, int32_t P0, int32_t P1, int lane, float4 *ring, int32_t *dring,
                     bool long_by_warp) {
    // keys from the one at P0 to the one at P1: key_rows keeps what starts in [P0, P1)
    const int32_t k_first = clampi(p.skey[P0], 0, p.R);
    const int32_t k_end = P1 < p.N ? clampi(p.skey[P1] + 1, k_first, p.R + 1) : p.R + 1;
    const int gs = min(8, p.seg_tile);
    const int gpt = p.seg_tile / gs;
    const bool split_on = p.seg_tile == kSegTile;
    const uint64_t src_pol = l2_evict_first_policy();
    for (int c0 = 0; c0 < p.D; c0 += 128) {
        const int col = c0 + lane * 4;
        const bool act = col < p.D;
        GroupCursor cur;
        cur.k_end = k_end;
        cur.P0 = P0;
        cur.P1 = P1;
        {
            int32_t st, en;
            load_seg(p, k_first, k_end, lane, st, en);
            cur.nst = cur.nen = 0;
            if (k_end - k_first > 32) load_seg(p, k_first + 32, k_end, lane, cur.nst, cur.nen);
            cur.R = key_rows(k_first, k_end, st, en, gs, split_on, P0, P1, lane);
            cur.q0 = 0;
        }
        Quad Qc, Qn;
        bool have = next_quad(p, cur, Qc, gs, gpt, split_on, lane);
        if (!have) continue;
        bool hn = next_quad(p, cur, Qn, gs, gpt, split_on, lane);
        int ji = 0;
        int issued = 0, consumed = 0;
        RowAcc ra;
        ra.F = ra.o = make_float4(0.f, 0.f, 0.f, 0.f);
        ra.tix = 0;
        GStack S;
        S.s0 = S.s1 = S.s2 = S.s3 = S.s4 = ra.F;
        auto issue_next = [&]() {
            if (have) {
                const int slot = issued % kStages;
                issue_group(p, ring + slot * kSlotF4, dring + slot * 2, Qc, ji, col, act, lane, src_pol);
                ++issued;
                if (++ji == Qc.n) {
                    ji = 0;
                    if (!hn) {
                        have = false;
                    } else {
                        Qc = Qn;
                        hn = next_quad(p, cur, Qn, gs, gpt, split_on, lane);
                    }
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int i = 0; i < kStages - 1; ++i) issue_next();
        while (consumed < issued) {
            issue_next();
            cp_async_wait<kStages - 1>();
            const int slot = consumed % kStages;
            consume_group(p, ring + slot * kSlotF4, dring + slot * 2, ra, S, gs, gpt, col, act, lane, long_by_warp);
            ++consumed;
        }
        cp_async_wait<0>();
    }
}

// Fold block: the ordered fold of the tile partials of split rows longer than
// kWarpFoldTiles tiles. The block waits (bounded) until every tile (in every
// column block) of the row is counted, stages the partials in shared memory
// with cp.async, kFoldTiles tiles per buffer in two buffers, and warp 0 folds
// them in ascending order.
constexpr int kFoldTiles = 192;

__device__ void fold_rows(const IdxParams &p, int first, int stride, int n_rows, float4 *stage) {
    __shared__ int timed_out;
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = first; i < n_rows; i += stride) {
        const int32_t k = clampi(p.heavy_rows[i], 0, p.R);
        const int32_t s0 = clampi(p.seg_start[k], 0, p.N), e0 = clampi(p.seg_start[k + 1], s0, p.N);
        const int32_t T = static_cast<int32_t>((e0 - s0 + kSegTile - 1) / kSegTile);
        if (tid == 0) {
            timed_out = wait_counter_geq(&p.tickets[k], T * ((p.D + 127) / 128)) ? 0 : 1;
            if (timed_out) record_error(p.hdr, DGR_ERR_TIMEOUT, 2);
        }
        __syncthreads();
        const bool skip = timed_out != 0;
        __syncthreads();
        if (skip) continue;
        for (int c0 = 0; c0 < p.D; c0 += 128) {
            const int w4 = min(32, (p.D - c0) / 4);  // float4 per tile row in this column block
            auto issue = [&](int buf, int32_t t0) {
                for (int e = tid; e < kFoldTiles * 32; e += kSegThreads) {
                    const int32_t t = t0 + e / 32;
                    const int c = e % 32;
                    if (t < T && c < w4)
                        cp_async16(stage + (buf * kFoldTiles + e / 32) * 32 + c,
                                   tile_slot(p, s0 + static_cast<int64_t>(t) * kSegTile, t == 0, c0 + c * 4));
                }
                cp_async_commit();
            };
            issue(0, 0);
            issue(1, kFoldTiles);
            float4 F = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int32_t t0 = 0, j = 0; t0 < T; t0 += kFoldTiles, ++j) {
                cp_async_wait<1>();
                __syncthreads();
                if (tid < 32 && lane < w4) {
                    const float4 *sb = stage + (j & 1) * kFoldTiles * 32;
                    const int nt = min(kFoldTiles, T - t0);
                    for (int u = 0; u < nt; ++u) F = (t0 + u == 0) ? sb[u * 32 + lane] : f4add(F, sb[u * 32 + lane]);
                }
                __syncthreads();
                issue(j & 1, t0 + 2 * kFoldTiles);
            }
            cp_async_wait<0>();
            if (tid < 32 && lane < w4) add_out(p, k, c0 + lane * 4, F);
            __syncthreads();
        }
        if (tid == 0) p.tickets[k] = 0;
    }
}

// Persistent: one block of 16 warps per SM. The first blocks (up to
// kMaxFoldBlocks, one per long split row) fold; every other warp takes an
// equal share of the sorted order.
__global__ void __launch_bounds__(kSegThreads, 1) segsum_kernel(const IdxParams p) {
    extern __shared__ __align__(16) float4 seg_smem[];
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    __shared__ int32_t s_good;
    if (threadIdx.x == 0) s_good = tag_ok(p);  // read while the previous launch finishes
    grid_dep_wait();
    __syncthreads();
    if (!s_good) return;  // hist refused the workspace: nothing is written
    {  // what the sort passes leave behind, cleared for the next call
        const int64_t tiles = static_cast<int64_t>(p.nb) * kDigits;
        const int64_t g = static_cast<int64_t>(blockIdx.x) * kSegThreads + threadIdx.x;
        for (int64_t i = g; i < tiles; i += static_cast<int64_t>(gridDim.x) * kSegThreads) {
            p.cnt[tiles + i] = 0;   // pass 1's tile counts (added up by pass 0)
            p.incl[tiles + i] = 0;  // pass 1's inclusive words
        }
        if (g < 2 * kDigits) p.hist[g] = 0;
    }
    if (p.D == 0) return;
    const int n_fold_rows = p.seg_tile == kSegTile ? clampi(p.hdr->pad[3], 0, p.max_fold_rows) : 0;
    const int n_fold = min(n_fold_rows, min(kMaxFoldBlocks, static_cast<int>(gridDim.x) - 1));
    if (static_cast<int>(blockIdx.x) < n_fold) {
        fold_rows(p, blockIdx.x, n_fold, n_fold_rows, seg_smem);
        return;
    }
    const int64_t W = static_cast<int64_t>(gridDim.x - n_fold) * kSegWarps;
    // shares handed to warps in the schedule's order (the warp count is known here only)
    const Sched sw = sched_over(p.sched_warps, static_cast<uint32_t>(W));
    const int64_t w = sched_item(sw, static_cast<uint32_t>((blockIdx.x - n_fold) * kSegWarps + wi));
    int64_t span = (static_cast<int64_t>(p.N) + W - 1) / W;
    if (span < 32) span = 32;
    const int64_t P0 = w * span;
    if (P0 >= p.N) return;
    const int32_t P1 = static_cast<int32_t>(min(P0 + span, static_cast<int64_t>(p.N)));
    float4 *ring = seg_smem + wi * (kStages * kSlotF4);
    int32_t *dring = reinterpret_cast<int32_t *>(seg_smem + kSegWarps * kStages * kSlotF4) + wi * (kStages * 2);
    walk(p, static_cast<int32_t>(P0), P1, lane, ring, dring, n_fold == 0);
}

static_assert(2 * kFoldTiles * 32 * 16 <= kSegSmemBytes, "fold stage fits the segsum shared memory");
struct IdxLayout {
    int32_t nb, n_pblk, max_fold_rows;
    size_t keys_a, vals_a, perm, skey, hist, count, cnt, incl, seg_start, tickets, slots, heavy, total;
};

IdxLayout idx_layout(int64_t N, int64_t R, int64_t D) {
    IdxLayout L{};
    L.nb = static_cast<int32_t>((N + kSortTile - 1) / kSortTile);
    L.n_pblk = static_cast<int32_t>((N + 127) / 128);
    L.max_fold_rows = static_cast<int32_t>(N / (kWarpFoldTiles * kSegTile + 1) + 1);
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
    L.hist = take(2 * kDigits * 4);
    L.count = take((R + 1) * 4);
    L.cnt = take(static_cast<size_t>(2) * L.nb * kDigits * 4);
    L.incl = take(static_cast<size_t>(2) * L.nb * kDigits * 4);
    L.seg_start = take((R + 2) * 4);
    L.tickets = take((R + 1) * 4);
    L.heavy = take(static_cast<size_t>(L.max_fold_rows) * 4);
    // last: the only region whose size depends on D, so a workspace for
    // (N, R, D) has the layout of (N, R, D') for every D' <= D
    L.slots = take(static_cast<size_t>(L.n_pblk) * 2 * D * 4);
    L.total = o;
    return L;
}

// Launch that may overlap the previous launch's tail on the stream (the kernel
// waits for it with grid_dep_wait before touching its results).
template <typename Kernel>
cudaError_t launch_after(Kernel kernel, unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                         const IdxParams &p) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
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
    p.n_buckets = static_cast<int32_t>((R + 1 + kDigits - 1) / kDigits);
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
    p.count = reinterpret_cast<int32_t *>(w + L.count);
    p.cnt = reinterpret_cast<int32_t *>(w + L.cnt);
    p.incl = reinterpret_cast<int32_t *>(w + L.incl);
    p.seg_start = reinterpret_cast<int32_t *>(w + L.seg_start);
    p.tickets = reinterpret_cast<int32_t *>(w + L.tickets);
    p.slots = reinterpret_cast<float *>(w + L.slots);
    p.heavy_rows = reinterpret_cast<int32_t *>(w + L.heavy);
    p.max_fold_rows = L.max_fold_rows;
    // segsum's fold blocks wait for tiles summed by other blocks: its grid is
    // the SMs usable at once (one block each), so every block is resident
    int sms = 0;
    dgr_status us = usable_sms(&sms);
    if (us != DGR_OK) return us;
    if (cudaFuncSetAttribute(segsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSegSmemBytes) != cudaSuccess)
        return DGR_ERR_CUDA;
    // pass 1 also has one item per 256-key bucket, where there are more buckets than tiles
    const unsigned pass1_items = static_cast<unsigned>(L.nb > p.n_buckets ? L.nb : p.n_buckets);
    p.sched_tiles = sched_for(static_cast<uint32_t>(L.nb));
    p.sched_pass1 = sched_for(pass1_items);
    p.sched_warps = sched_setting();
    hist_kernel<<<sched_grid(static_cast<unsigned>(L.nb)), kSortThreads, 0, s>>>(p);
    // segsum (persistent: one block per SM, each warp one share of the sorted
    // order) runs even without columns: it clears the sort's counters
    if (launch_after(pass_kernel<0>, sched_grid(static_cast<unsigned>(L.nb)), kPassThreads, 0, s, p) != cudaSuccess ||
        launch_after(pass_kernel<1>, sched_grid(pass1_items), kPassThreads, 0, s, p) != cudaSuccess ||
        launch_after(segsum_kernel, static_cast<unsigned>(sms), kSegThreads, kSegSmemBytes, s, p) != cudaSuccess)
        return DGR_ERR_CUDA;
    return launch_status();
}
