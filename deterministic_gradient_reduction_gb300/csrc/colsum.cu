// Ordered column sum: out[h] = fold_j pw_W(x[t][h] : t in tile j).
//
// Megatron-LM PR #8244 (ordered reduction for the fused pre-GDR gate
// backward), description: every program writes its own FP32 partial sums and
// the caller reduces them in order on the same stream. Here both halves run in
// ONE launch:
//   - producer CTAs, one per (tile of W tokens, block of columns): 16-byte
//     vector loads, the pairwise tree of the tile (in registers over the rows a
//     thread owns, then across threads in shared memory, always over aligned
//     sub-windows so the tree is exactly the canonical one), one FP32 slot row
//     per tile, then an increment of the ready counter of its group of 32
//     tiles;
//   - folder CTAs (the first blockIdx values), one per block of FC columns
//     (4 for H <= 256, at most 64 folders):
//     they wait (bounded) for each batch of tiles to be ready, stage the slots
//     through shared memory with many loader warps, and fold them in ascending
//     tile order on one thread per column. The fold overlaps the stream, so a
//     long dependent chain of adds (65,536 tiles for 1 GiB of bf16 at H = 64)
//     hides under the HBM time instead of following it.
// Each slot word says itself whether it has been written: a partial is stored
// as the complement of its bits (0 = empty), and the folder zeroes the words
// it consumes. So no producer fences its slot writes before the count: the
// counters only tell the folder when to look, and a word the folder reads
// before its write has arrived is read again (bounded). Producers never wait,
// so the folders' waits always end.
#include "dgr_common.cuh"
#include "dgr_diag.h"

namespace dgr {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpThreads = 512;                 // warp-producer kernel: one CTA per SM
constexpr int kWarpSmemBytes = 116 * 1024;        // more than half an SM: one CTA per SM
constexpr int kGroupTiles = 32;                 // tiles per ready counter
constexpr int kFolderSmemBytes = 32 * 1024;     // double-buffered slot batches (<= 1024 tiles each)
constexpr int kMaxFolders = 64;

struct ColsumParams {
    const char *x;
    int64_t stride_b, stride_s;  // elements
    int32_t S;
    int32_t T;
    int32_t H;
    int32_t W;                   // tile rows (power of two)
    int32_t n_tiles;
    int32_t flat;                // tokens are at t * stride_s
    // producer mapping
    int32_t RG, CB, V, n_pcb, TPC;
    // 1: warp producers (one warp per tile)
    int32_t stream_mode;
    // folder mapping
    int32_t FC, n_fcb, batch;
    float *out;
    int32_t accumulate;
    float *slots;                // [H][col_stride] (tile fastest)
    int64_t col_stride;
    int32_t *counters;           // [n_groups]
    WsHeader *hdr;
    // folder CTAs of this launch (the first blockIdx values): all of them when
    // folders and producers share one launch, none in a producers-only launch
    int32_t fold_ctas;
    int32_t n_units;             // producer work units (tiles, or tile groups x column blocks)
    Sched sched;                 // which producer takes which unit
};

template <int DT>
struct Elem;
template <>
struct Elem<DGR_DTYPE_BF16> {
    static constexpr int kSize = 2;
    static __device__ __forceinline__ float load1(const char *p) {
        return bf16_bits_to_f32(*reinterpret_cast<const uint16_t *>(p));
    }
    static __device__ __forceinline__ void unpack(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
template <>
struct Elem<DGR_DTYPE_F32> {
    static constexpr int kSize = 4;
    static __device__ __forceinline__ float load1(const char *p) {
        return *reinterpret_cast<const float *>(p);
    }
    static __device__ __forceinline__ void unpack(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
};

// Slots are column-major inside each folder block: column c of tile j is at
// c * col_stride + j (col_stride = n_tiles rounded up to 4), so a folder reads
// four consecutive tiles of its column with one 16-byte load.
__device__ __forceinline__ int64_t slot_index(const ColsumParams &p, int c, int j) {
    return static_cast<int64_t>(c) * p.col_stride + j;
}

// Slot words: the complement of the partial's bits, so that 0 means "not
// written yet". The one partial whose complement is 0 (the NaN with every bit
// set) is stored as the NaN next to it, which can change a NaN's payload and
// nothing else.
__device__ __forceinline__ uint32_t slot_word(float v) {
    const uint32_t w = ~__float_as_uint(v);
    return w != 0u ? w : 1u;
}
__device__ __forceinline__ float slot_value(uint32_t w) { return __uint_as_float(~w); }

__device__ __forceinline__ void st_slot(const ColsumParams &p, int c, int j, float v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p.slots + slot_index(p, c, j)), "r"(slot_word(v))
                 : "memory");
}

__device__ __forceinline__ uint4 ld_slot4(const float *a) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(a)
                 : "memory");
    return v;
}

// The first n (1..4) words of a slot quad, all written: read again until
// none is 0, at most kWaitLimitNs. Returns false on timeout.
__device__ __noinline__ bool wait_slot4(const float *a, int n, uint4 &v) {
    const uint64_t t0 = globaltimer_ns();
    unsigned ns = 32;
    while (true) {
        const bool ready = v.x != 0u && (n < 2 || v.y != 0u) && (n < 3 || v.z != 0u) && (n < 4 || v.w != 0u);
        if (ready) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        __nanosleep(ns);
        if (ns < 1024) ns <<= 1;
        v = ld_slot4(a);
    }
}

__device__ __forceinline__ int64_t token_offset(const ColsumParams &p, int32_t t) {
    if (p.flat) return static_cast<int64_t>(t) * p.stride_s;
    const int32_t b = t / p.S;
    const int32_t s = t - b * p.S;
    return static_cast<int64_t>(b) * p.stride_b + static_cast<int64_t>(s) * p.stride_s;
}

// One producer unit: TPC consecutive tiles (a group of RG*CB threads each)
// for column vectors [cv0, cv0 + CB). VE = elements per vector (8 bf16 or 4
// fp32 for 16-byte loads, 1 for the scalar path); RPT = rows a thread owns.
// A thread keeps its RPT rows in flight as raw 16-byte words and widens them
// pair by pair into the first tree level.
template <int DT, int VE, int RPT>
__device__ void produce(const ColsumParams &p, int unit, float *sm) {
    using E = Elem<DT>;
    const int tg = unit / p.n_pcb;                 // tile group
    const int pcb = unit - tg * p.n_pcb;
    const int tid = threadIdx.x;
    const int tpt = p.RG * p.CB;                   // threads per tile
    const int ts = tid / tpt;                      // tile slot in this CTA
    const int tt = tid - ts * tpt;
    const int g = tt / p.CB;                       // row group
    const int v = tt - g * p.CB;                   // column vector within the block
    const int j = tg * p.TPC + ts;                 // tile
    const int cv0 = pcb * p.CB;
    const int cb_here = min(p.CB, p.V - cv0);
    const bool active = ts < p.TPC && j < p.n_tiles && v < cb_here;
    const int64_t t0 = static_cast<int64_t>(j) * p.W;
    const int count = active ? static_cast<int>(min(static_cast<int64_t>(p.W), p.T - t0)) : 0;
    const int groups_present = (count + RPT - 1) / RPT;
    const int nrows = active ? max(0, min(RPT, count - g * RPT)) : 0;
    float *tsm = sm + ts * tpt * VE;

    if (nrows > 0) {
        const int c0 = (cv0 + v) * VE;
        constexpr int RW = VE == 1 ? 1 : 4;        // 32-bit words per vector
        uint32_t raw[RPT][RW];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            if (r < nrows) {
                const int32_t t = static_cast<int32_t>(t0) + g * RPT + r;
                const char *src = p.x + (token_offset(p, t) + c0) * E::kSize;
                if constexpr (VE == 1) {
                    raw[r][0] = __float_as_uint(E::load1(src));
                } else {
                    const uint4 q = ldg_nc_v4(src);
                    raw[r][0] = q.x; raw[r][1] = q.y; raw[r][2] = q.z; raw[r][3] = q.w;
                }
            }
        }
        // level 1 while widening: rows (2i, 2i+1)
        constexpr int NP = RPT > 1 ? RPT / 2 : 1;
        float pr[NP][VE];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int r = 2 * i;
            if (r < nrows) {
                float a[VE];
                if constexpr (VE == 1) a[0] = __uint_as_float(raw[r][0]);
                else E::unpack(make_uint4(raw[r][0], raw[r][1], raw[r][2], raw[r][3]), a);
                if (RPT > 1 && r + 1 < nrows) {
                    float b[VE];
                    if constexpr (VE == 1) b[0] = __uint_as_float(raw[r + 1][0]);
                    else E::unpack(make_uint4(raw[r + 1][0], raw[r + 1][1], raw[r + 1][2], raw[r + 1][3]), b);
#pragma unroll
                    for (int e = 0; e < VE; ++e) a[e] = __fadd_rn(a[e], b[e]);
                }
#pragma unroll
                for (int e = 0; e < VE; ++e) pr[i][e] = a[e];
            }
        }
        // levels 2.. in registers: aligned windows of 2s pairs
        const int npresent = (nrows + 1) / 2;
#pragma unroll
        for (int s = 1; s < NP; s *= 2) {
#pragma unroll
            for (int i = 0; i + s < NP; i += 2 * s) {
                if (i + s < npresent) {
#pragma unroll
                    for (int e = 0; e < VE; ++e) pr[i][e] = __fadd_rn(pr[i][e], pr[i + s][e]);
                }
            }
        }
        float *dst = tsm + (g * p.CB + v) * VE;
#pragma unroll
        for (int e = 0; e < VE; ++e) dst[e] = pr[0][e];
    }
    __syncthreads();
    // shared-memory levels: row group g absorbs g + s when both are present
    for (int s = 1; s < p.RG; s *= 2) {
        if (active && (g % (2 * s)) == 0 && g + s < groups_present) {
            float *a = tsm + (g * p.CB + v) * VE;
            const float *b = tsm + ((g + s) * p.CB + v) * VE;
#pragma unroll
            for (int e = 0; e < VE; ++e) a[e] = __fadd_rn(a[e], b[e]);
        }
        __syncthreads();
    }
    if (active && g == 0) {
        const float *root = tsm + v * VE;
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            const int c = (cv0 + v) * VE + e;
            if (c < p.H) st_slot(p, c, j, root[e]);
        }
    }
    __syncthreads();
    if (tid == 0) {
        // the CTA's tiles lie in one group of 32 (TPC divides 32)
        const int first = tg * p.TPC;
        const int n_here = min(p.TPC, p.n_tiles - first);
        atomicAdd(&p.counters[first / kGroupTiles], n_here);
    }
}

// Warp producers (vector loads, V column vectors with V dividing 32): one warp
// per tile. Lane = (row group, vector): RGW = 32 / V row groups of RPL = W /
// RGW consecutive rows each. A lane sums its rows by the tree's first levels
// in registers (batches of up to 16 raw 16-byte words in flight, a binary
// counter over the batches), and the remaining levels are xor-shuffles
// between row groups at lane distance V, 2V, ... - aligned windows, so the
// tree is exactly the canonical one, with no shared memory and no block
// barrier. Lanes of row group 0 then hold the tile partial.
// The tile's slot row is written here; its ready count is left to the
// caller (publish_tile), which issues it once the warp's next tile has its
// first loads in flight. `pending` is the warp's previous unpublished tile
// (-1: none).
__device__ __forceinline__ void publish_tile(const ColsumParams &p, int pending) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) atomicAdd(&p.counters[pending / kGroupTiles], 1);
}

// MAXB: raw 16-byte loads a lane keeps in flight (a batch); the tree is the
// same for any batch size (batches are aligned subtrees of the tile).
template <int DT, int VE, int RPL, int MAXB = 8>
__device__ __forceinline__ void produce_warp_tile(const ColsumParams &p, int64_t wunit, int pending) {
    using E = Elem<DT>;
    constexpr int BATCH = RPL < MAXB ? RPL : MAXB;
    constexpr int NB = RPL / BATCH;  // batches, a power of two <= 16
    constexpr int LV = NB >= 16 ? 4 : NB >= 8 ? 3 : NB >= 4 ? 2 : NB >= 2 ? 1 : 0;
    const int lane = threadIdx.x & 31;
    if (wunit >= p.n_tiles) {
        if (pending >= 0) publish_tile(p, pending);
        return;
    }
    const int j = static_cast<int>(wunit);
    const int V = p.V;
    const int g = lane / V;
    const int v = lane - g * V;
    const int64_t t0 = static_cast<int64_t>(j) * p.W;
    const int count = static_cast<int>(min(static_cast<int64_t>(p.W), p.T - t0));
    const int nrows = max(0, min(RPL, count - g * RPL));
    const int c0 = v * VE;
    float stack[LV + 1][VE];
    float acc[VE];
#pragma unroll
    for (int bi = 0; bi < NB; ++bi) {
        const int rb = bi * BATCH;  // first row of the batch within the lane's rows
        uint4 raw[BATCH];
#pragma unroll
        for (int r = 0; r < BATCH; ++r) {
            if (rb + r < nrows) {
                const int32_t t = static_cast<int32_t>(t0) + g * RPL + rb + r;
                raw[r] = ldg_nc_v4(p.x + (token_offset(p, t) + c0) * E::kSize);
            }
        }
        if (bi == 0 && pending >= 0) publish_tile(p, pending);
        // the batch's subtree (rows rb .. rb+BATCH-1), absent rows skipped;
        // level 1 is taken while widening, pair by pair
        const int nb_rows = max(0, min(BATCH, nrows - rb));
        constexpr int NP = BATCH > 1 ? BATCH / 2 : 1;
        float lv[NP][VE];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int r = 2 * i;
            if (r < nb_rows) {
                E::unpack(raw[r], lv[i]);
                if (BATCH > 1 && r + 1 < nb_rows) {
                    float b2[VE];
                    E::unpack(raw[r + 1], b2);
#pragma unroll
                    vadd<VE>(lv[i], lv[i], b2);
                }
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
    // ragged end: complete blocks of the set bits of the present batch count,
    // smallest first, each larger (earlier) block on the left
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
    // cross-lane levels: row group g absorbs g + s (lane distance s * V)
    bool present = nrows > 0;
    for (int s = 1; s * V < 32; s *= 2) {
        const bool left_is_me = (g & s) == 0;
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
    if (g == 0) {
#pragma unroll
        for (int e = 0; e < VE; ++e) st_slot(p, c0 + e, j, acc[e]);
    }
}

// One folder CTA: columns [f*FC, f*FC + FC), all tiles in ascending order.
// Shared memory holds two batches, column-major: buf[cc * batch + k].
__device__ void fold(const ColsumParams &p, int f, float *sm) {
    __shared__ int abort_flag;
    __shared__ int ticket;
    const int tid = threadIdx.x;
    const int chain_threads = ((p.FC + 31) / 32) * 32;
    const int nthreads = blockDim.x;
    const int loader_threads = nthreads - chain_threads;
    const int ltid = tid - chain_threads;  // loader index (>= 0 for loaders)
    const int n_batches = (p.n_tiles + p.batch - 1) / p.batch;
    const int col = f * p.FC + tid;
    if (tid == 0) abort_flag = 0;
    __syncthreads();

    // Loaders: wait for batch i's tile groups, then copy its slots to buffer i%2.
    auto load = [&](int i) {
        const int j0 = i * p.batch;
        const int j1 = min(j0 + p.batch, p.n_tiles);
        if (ltid < 32) {  // one lane per group of the batch (a batch spans <= 32 groups)
            const int grp = j0 / kGroupTiles + ltid;
            bool ok = true;
            if (grp <= (j1 - 1) / kGroupTiles) {
                const int tiles_in_group = min(kGroupTiles, p.n_tiles - grp * kGroupTiles);
                ok = wait_counter_geq(&p.counters[grp], tiles_in_group * p.n_pcb);
            }
            if (__any_sync(0xffffffffu, !ok)) {
                if (ltid == 0) {
                    record_error(p.hdr, DGR_ERR_TIMEOUT, 1);
                    abort_flag = 1;
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(loader_threads) : "memory");
        if (abort_flag) return;
        // the counts said the batch is written: its words are read (again,
        // bounded, where one has not arrived yet), decoded into shared memory
        // and zeroed for the next call
        const int q4 = (j1 - j0 + 3) / 4;  // float4 per column (the column stride is padded to 4)
        const int n4 = q4 * p.FC;
        float4 *d4 = reinterpret_cast<float4 *>(sm + (i & 1) * p.batch * p.FC);
        bool ok = true;
        for (int q = ltid; q < n4; q += loader_threads) {
            const int cc = q / q4;
            const int k4 = q - cc * q4;
            if (f * p.FC + cc >= p.H) continue;  // a column past H: never written, never folded
            float *s4 = p.slots + slot_index(p, f * p.FC + cc, j0) + 4 * k4;
            const int n = min(4, j1 - j0 - 4 * k4);  // words of real tiles (the stride pads to 4)
            uint4 v = ld_slot4(s4);
            const bool ready = v.x != 0u && (n < 2 || v.y != 0u) && (n < 3 || v.z != 0u) && (n < 4 || v.w != 0u);
            if (!ready && !wait_slot4(s4, n, v)) {
                ok = false;
                break;
            }
            d4[cc * (p.batch / 4) + k4] = make_float4(slot_value(v.x), slot_value(v.y), slot_value(v.z),
                                                      slot_value(v.w));
            *reinterpret_cast<uint4 *>(s4) = make_uint4(0u, 0u, 0u, 0u);
        }
        if (!ok) {
            record_error(p.hdr, DGR_ERR_TIMEOUT, 2);
            abort_flag = 1;
        }
    };

    if (ltid >= 0) load(0);
    __syncthreads();
    float F = 0.0f;
    for (int i = 0; i < n_batches; ++i) {
        if (abort_flag) break;
        if (ltid >= 0) {
            if (i + 1 < n_batches) load(i + 1);
        } else if (tid < p.FC && col < p.H) {
            const float4 *b4 = reinterpret_cast<const float4 *>(sm + (i & 1) * p.batch * p.FC + tid * p.batch);
            const int cnt = min(p.batch, p.n_tiles - i * p.batch);
            int k = 0;
            if (i == 0) {  // the fold starts from tile 0's partial
                const float4 q = b4[0];
                F = q.x;
                if (cnt > 1) F = __fadd_rn(F, q.y);
                if (cnt > 2) F = __fadd_rn(F, q.z);
                if (cnt > 3) F = __fadd_rn(F, q.w);
                k = 4;
            }
            // blocks of 16 tiles: the next block's four 16-byte loads are issued
            // before the current block's 16 dependent adds (the last block
            // reloads itself instead of reading past the batch)
            const int kfull = cnt > k ? k + ((cnt - k) / 16) * 16 : k;
            if (k < kfull) {
                float4 r0 = b4[(k >> 2)], r1 = b4[(k >> 2) + 1], r2 = b4[(k >> 2) + 2], r3 = b4[(k >> 2) + 3];
                for (; k < kfull; k += 16) {
                    const int nk = (k + 16 < kfull) ? k + 16 : k;
                    const float4 s0 = b4[(nk >> 2)], s1 = b4[(nk >> 2) + 1], s2 = b4[(nk >> 2) + 2],
                                 s3 = b4[(nk >> 2) + 3];
                    F = __fadd_rn(F, r0.x); F = __fadd_rn(F, r0.y); F = __fadd_rn(F, r0.z); F = __fadd_rn(F, r0.w);
                    F = __fadd_rn(F, r1.x); F = __fadd_rn(F, r1.y); F = __fadd_rn(F, r1.z); F = __fadd_rn(F, r1.w);
                    F = __fadd_rn(F, r2.x); F = __fadd_rn(F, r2.y); F = __fadd_rn(F, r2.z); F = __fadd_rn(F, r2.w);
                    F = __fadd_rn(F, r3.x); F = __fadd_rn(F, r3.y); F = __fadd_rn(F, r3.z); F = __fadd_rn(F, r3.w);
                    r0 = s0;
                    r1 = s1;
                    r2 = s2;
                    r3 = s3;
                }
            }
            for (; k + 4 <= cnt; k += 4) {
                const float4 q = b4[k >> 2];
                F = __fadd_rn(F, q.x);
                F = __fadd_rn(F, q.y);
                F = __fadd_rn(F, q.z);
                F = __fadd_rn(F, q.w);
            }
            if (k < cnt) {
                const float4 q = b4[k >> 2];
                F = __fadd_rn(F, q.x);
                if (k + 1 < cnt) F = __fadd_rn(F, q.y);
                if (k + 2 < cnt) F = __fadd_rn(F, q.z);
            }
        }
        __syncthreads();
    }
    if (abort_flag) return;
    if (tid < p.FC && col < p.H) p.out[col] = p.accumulate ? __fadd_rn(p.out[col], F) : F;

    // The last folder to finish resets the ready counters for the next call:
    // every producer has published by now (all groups were consumed).
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        ticket = atomicAdd(&p.hdr->pad[0], 1);
    }
    __syncthreads();
    if (ticket == p.n_fcb - 1) {
        const int n_groups = (p.n_tiles + kGroupTiles - 1) / kGroupTiles;
        for (int q = tid; q < n_groups; q += nthreads) p.counters[q] = 0;
        if (tid == 0) p.hdr->pad[0] = 0;
    }
}

// Folder blocks f of this launch's folder CTAs (a CTA takes several when the
// launch has fewer folder CTAs than folder blocks).
__device__ __forceinline__ void fold_all(const ColsumParams &p, float *sm) {
    for (int f = blockIdx.x; f < p.n_fcb; f += p.fold_ctas) fold(p, f, sm);
}

template <int DT, int VE, int RPT>
__global__ void __launch_bounds__(kThreads) colsum_kernel(const ColsumParams p) {
    extern __shared__ __align__(128) float smem[];
    if (static_cast<int>(blockIdx.x) < p.fold_ctas) {
        fold_all(p, smem);
    } else {
        const int n_prod = static_cast<int>(gridDim.x) - p.fold_ctas;
        for (int u = blockIdx.x - p.fold_ctas; u < p.n_units; u += n_prod)
            produce<DT, VE, RPT>(p, static_cast<int>(sched_item(p.sched, static_cast<uint32_t>(u))), smem);
    }
}

// The same with warp producers. One 512-thread CTA per SM (the launch asks
// for more than half an SM's shared memory), so a folder has its SM to
// itself: its chain of dependent adds then issues at the add latency instead
// of competing with producer warps for issue slots. Producer CTAs are
// persistent; warp w of all producer warps takes tiles w, w + n, w + 2n, ...
template <int DT, int VE, int RPL>
__global__ void __launch_bounds__(kWarpThreads, 1) colsum_warp_kernel(const ColsumParams p) {
    extern __shared__ __align__(128) float smem[];
    if (static_cast<int>(blockIdx.x) < p.fold_ctas) {
        fold_all(p, smem);
    } else {
        const int64_t wpc = kWarpThreads / 32;
        const int64_t n_warps = static_cast<int64_t>(gridDim.x - p.fold_ctas) * wpc;
        int pending = -1;
        for (int64_t w = static_cast<int64_t>(blockIdx.x - p.fold_ctas) * wpc + (threadIdx.x >> 5); w < p.n_tiles;
             w += n_warps) {
            const int tile = static_cast<int>(sched_item(p.sched, static_cast<uint32_t>(w)));
            produce_warp_tile<DT, VE, RPL>(p, tile, pending);
            pending = tile;
        }
        if (pending >= 0) publish_tile(p, pending);
    }
}

// Small inputs (at most kSmallTiles tiles): one warp per tile writes its
// slot row and takes an integer ticket; the warp that takes the last ticket
// folds every column over the tiles in ascending order and writes out. No
// folder CTA, no waiting.
constexpr int kSmallTiles = 512;
constexpr int kSmallWarps = 4;

template <int DT, int VE, int RPL>
__global__ void __launch_bounds__(kSmallWarps * 32) colsum_small_kernel(const ColsumParams p) {
    const int lane = threadIdx.x & 31;
    const int nw = static_cast<int>(gridDim.x) * kSmallWarps;
    bool last = false;
    // tiles in the schedule's order; with a capped grid a warp takes several
    for (int w = static_cast<int>(blockIdx.x) * kSmallWarps + (threadIdx.x >> 5); w < p.n_tiles && !last; w += nw) {
        produce_warp_tile<DT, VE, RPL, 16>(p, static_cast<int>(sched_item(p.sched, static_cast<uint32_t>(w))), -1);
        __threadfence();  // this lane's slot-row writes before the ticket
        __syncwarp();
        int t = 0;
        if (lane == 0) t = atomicAdd(&p.hdr->pad[0], 1);
        last = __shfl_sync(0xffffffffu, t, 0) == p.n_tiles - 1;
    }
    if (!last) return;
    __threadfence();  // every other warp's slot rows are visible after its ticket
    const int n4 = (p.n_tiles + 3) / 4;  // 16-byte groups of 4 tiles per column (the stride is padded to 4)
    for (int c = lane; c < p.H; c += 32) {
        uint4 *s4 = reinterpret_cast<uint4 *>(p.slots + slot_index(p, c, 0));
        float F = 0.0f;
        for (int q0 = 0; q0 < n4; q0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (q0 + u < n4) v[u] = __ldcg(s4 + q0 + u);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (q0 + u < n4) s4[q0 + u] = make_uint4(0u, 0u, 0u, 0u);  // empty again for the next call
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (q0 + u >= n4) break;
                const int k = 4 * (q0 + u);
                const float e[4] = {slot_value(v[u].x), slot_value(v[u].y), slot_value(v[u].z), slot_value(v[u].w)};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (k + i < p.n_tiles) F = (k + i == 0) ? e[i] : __fadd_rn(F, e[i]);
            }
        }
        p.out[c] = p.accumulate ? __fadd_rn(p.out[c], F) : F;
    }
    if (lane == 0) p.hdr->pad[0] = 0;
}

using ColsumKernel = void (*)(const ColsumParams);

template <int DT, int VE>
ColsumKernel cta_kernel(int rpt) {
    switch (rpt) {
        case 1: return colsum_kernel<DT, VE, 1>;
        case 2: return colsum_kernel<DT, VE, 2>;
        case 4: return colsum_kernel<DT, VE, 4>;
        case 8: return colsum_kernel<DT, VE, 8>;
        case 16: return colsum_kernel<DT, VE, 16>;
        default: return nullptr;
    }
}

template <int DT, int VE>
ColsumKernel warp_kernel(int rpl) {
    switch (rpl) {
        case 2: return colsum_warp_kernel<DT, VE, 2>;
        case 4: return colsum_warp_kernel<DT, VE, 4>;
        case 8: return colsum_warp_kernel<DT, VE, 8>;
        case 16: return colsum_warp_kernel<DT, VE, 16>;
        case 32: return colsum_warp_kernel<DT, VE, 32>;
        case 64: return colsum_warp_kernel<DT, VE, 64>;
        case 128: return colsum_warp_kernel<DT, VE, 128>;
        default: return nullptr;
    }
}

template <int DT, int VE>
ColsumKernel small_kernel(int rpl) {
    switch (rpl) {
        case 2: return colsum_small_kernel<DT, VE, 2>;
        case 4: return colsum_small_kernel<DT, VE, 4>;
        case 8: return colsum_small_kernel<DT, VE, 8>;
        case 16: return colsum_small_kernel<DT, VE, 16>;
        case 32: return colsum_small_kernel<DT, VE, 32>;
        case 64: return colsum_small_kernel<DT, VE, 64>;
        case 128: return colsum_small_kernel<DT, VE, 128>;
        default: return nullptr;
    }
}

// How a call is launched.
//   path 0: at most kSmallTiles warp-producer tiles: one launch, a ticket,
//           the last warp folds (nothing waits);
//   path 1: warp producers (persistent, one CTA per SM) and folder CTAs;
//   path 2: CTA producers (one per unit) and folder CTAs.
// On paths 1 and 2 the folders wait for the producers, so one launch holds
// both only when every folder CTA and at least one producer CTA can be
// resident at once; otherwise the producers run in a first launch and the
// folders, which then find every tile written, in a second.
struct ColsumPlan {
    int32_t path, launches;
    int64_t prod_ctas;  // producer CTAs (path 0: CTAs of kSmallWarps warps)
    int32_t fold_ctas;  // folder CTAs (in the one launch, or in the second)
};

ColsumPlan colsum_plan(int32_t n_tiles, int32_t n_fcb, int64_t n_units, bool warp_producers, int32_t sms,
                       int32_t cta_occupancy, int32_t cap) {
    ColsumPlan pl{};
    auto capped = [cap](int64_t g) { return (cap > 0 && g > cap) ? static_cast<int64_t>(cap) : g; };
    if (warp_producers && n_tiles <= kSmallTiles) {
        pl.path = 0;
        pl.launches = 1;
        pl.prod_ctas = capped((n_tiles + kSmallWarps - 1) / kSmallWarps);
        return pl;
    }
    if (warp_producers) {
        pl.path = 1;
        const int64_t need = (n_tiles + kWarpThreads / 32 - 1) / (kWarpThreads / 32);
        const int64_t resident = capped(sms);  // one CTA per SM
        if (resident >= n_fcb + 1) {
            pl.launches = 1;
            pl.prod_ctas = need < resident - n_fcb ? need : resident - n_fcb;
            pl.fold_ctas = n_fcb;
        } else {
            pl.launches = 2;
            pl.prod_ctas = need < resident ? need : (resident > 0 ? resident : 1);
            pl.fold_ctas = static_cast<int32_t>(n_fcb < resident ? n_fcb : (resident > 0 ? resident : 1));
        }
        return pl;
    }
    pl.path = 2;
    const int64_t slots = static_cast<int64_t>(sms) * (cta_occupancy > 0 ? cta_occupancy : 1);
    if (slots >= n_fcb + 1 && (cap == 0 || cap >= n_fcb + 1)) {
        pl.launches = 1;
        pl.fold_ctas = n_fcb;
        pl.prod_ctas = cap > 0 && n_units > cap - n_fcb ? cap - n_fcb : n_units;
    } else {
        pl.launches = 2;
        pl.prod_ctas = capped(n_units);
        pl.fold_ctas = static_cast<int32_t>(capped(n_fcb));
    }
    return pl;
}

struct Layout {
    int32_t n_tiles, n_groups, FC, n_fcb;
    int64_t col_stride;
    size_t counters_off, slots_off, total;
};

Layout colsum_layout(int64_t T, int64_t H, int32_t W) {
    Layout L{};
    L.n_tiles = static_cast<int32_t>((T + W - 1) / W);
    L.n_groups = (L.n_tiles + kGroupTiles - 1) / kGroupTiles;
    // FC columns per folder, a multiple of 4 (float4 staging): 4 for H <= 256
    const int64_t fcb4 = (H + 3) / 4;
    L.FC = static_cast<int32_t>(4 * ((fcb4 + kMaxFolders - 1) / kMaxFolders));
    if (L.FC < 4) L.FC = 4;
    L.n_fcb = static_cast<int32_t>((H + L.FC - 1) / L.FC);
    L.counters_off = sizeof(WsHeader);
    L.slots_off = L.counters_off + align_up(static_cast<size_t>(L.n_groups) * 4);
    L.col_stride = (static_cast<int64_t>(L.n_tiles) + 3) / 4 * 4;
    L.total = L.slots_off + align_up(static_cast<size_t>(L.n_fcb) * L.FC * L.col_stride * 4);
    return L;
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" size_t dgr_colsum_workspace_bytes(int64_t T, int64_t H, int32_t tile_rows) {
    if (T < 0 || H < 0 || H > 4096 || T > INT32_MAX || !is_pow2(tile_rows) || tile_rows > 4096) return 0;
    return colsum_layout(T, H, tile_rows).total;
}

namespace dgr {
namespace {

// Argument checks shared by both entry points (the workspace's own checks are
// the caller's). `nothing` is set when H = 0: there is nothing to do.
dgr_status colsum_args(const void *x, int32_t dtype, int64_t B, int64_t S, int64_t H, int64_t stride_b,
                       int64_t stride_s, const float *out, int32_t tile_rows, bool &nothing) {
    nothing = false;
    if (dtype != DGR_DTYPE_BF16 && dtype != DGR_DTYPE_F32) return DGR_ERR_INVALID_ARG;
    if (B < 0 || S < 0 || H < 0 || stride_b < 0 || stride_s < 0) return DGR_ERR_INVALID_ARG;
    if (!is_pow2(tile_rows) || tile_rows > 4096) return DGR_ERR_INVALID_ARG;
    if (H > 4096 || (S > 0 && B > INT32_MAX / S)) return DGR_ERR_UNSUPPORTED;
    if (H == 0) {
        nothing = true;
        return DGR_OK;
    }
    if (!out || (B * S > 0 && !x)) return DGR_ERR_INVALID_ARG;
    if (!aligned(out, 4)) return DGR_ERR_MISALIGNED;
    return DGR_OK;
}

// The input's alignment and its overlap with out.
dgr_status colsum_input_checks(const void *x, int32_t dtype, int64_t B, int64_t S, int64_t H, int64_t stride_b,
                               int64_t stride_s, const float *out) {
    const int esize = dtype == DGR_DTYPE_BF16 ? 2 : 4;
    const int64_t T = B * S;
    if (x && !aligned(x, esize)) return DGR_ERR_MISALIGNED;
    const int64_t x_extent = T > 0 ? ((B - 1) * stride_b + (S - 1) * stride_s + H) * esize : 0;
    if (ranges_overlap(out, H * 4, x, x_extent)) return DGR_ERR_ALIAS;
    return DGR_OK;
}

// Producer geometry: vector width VE (elements per 16-byte load, 1 for the
// scalar path), column vectors V, the CTA producers' mapping (CB vectors and
// RG row groups of rpt rows per tile, TPC tiles per CTA, n_pcb column blocks)
// and, for power-of-two V, the warp producers' rows per lane rpl.
void colsum_geometry(ColsumParams &p, int64_t H, int32_t tile_rows, int esize, bool vec_ok, int32_t n_tiles,
                     int &VE, int &rpt, int &rpl) {
    const int vec = 16 / esize;
    VE = vec_ok ? vec : 1;
    p.V = static_cast<int32_t>((H + VE - 1) / VE);
    p.CB = p.V < 32 ? p.V : 32;
    // each thread owns up to 16 rows; a tile takes RG * CB threads and a CTA
    // packs TPC tiles (a power of two dividing the 32-tile counter group)
    rpt = tile_rows < 16 ? tile_rows : 16;
    if ((tile_rows / rpt) * p.CB > kThreads) p.CB = kThreads / (tile_rows / rpt);
    p.RG = tile_rows / rpt;
    p.n_pcb = (p.V + p.CB - 1) / p.CB;
    int tpc = 1;
    const int64_t units_min = 4LL * 152;  // keep enough CTAs to fill the GPU
    while (tpc < 32 && 2 * tpc * p.RG * p.CB <= kThreads &&
           (static_cast<int64_t>(n_tiles) + 2 * tpc - 1) / (2 * tpc) * p.n_pcb >= units_min)
        tpc *= 2;
    if (n_tiles <= 32) {  // tiny inputs: as few CTAs as the threads allow
        while (tpc < 32 && 2 * tpc * p.RG * p.CB <= kThreads && tpc < n_tiles) tpc *= 2;
    }
    p.TPC = tpc;
    // Warp producers when a power-of-two number of 16-byte column vectors
    // (at most 32) tiles a warp and each lane gets 2 .. 128 rows.
    p.stream_mode = 0;
    rpl = 0;
    if (vec_ok && p.V <= 32 && (p.V & (p.V - 1)) == 0) {
        rpl = static_cast<int>(static_cast<int64_t>(tile_rows) * p.V / 32);
        if (rpl >= 2 && rpl <= 128) p.stream_mode = 1;
    }
}

// Enqueues the call on `stream` once every argument has been checked; ws holds
// at least colsum_layout(B*S, H, tile_rows).total zeroed bytes.
dgr_status colsum_enqueue(const void *x, int32_t dtype, int64_t B, int64_t S, int64_t H, int64_t stride_b,
                          int64_t stride_s, float *out, int32_t accumulate, int32_t tile_rows, void *ws,
                          void *stream) {
    const int64_t T = B * S;
    const Layout L = colsum_layout(T, H, tile_rows);
    const int esize = dtype == DGR_DTYPE_BF16 ? 2 : 4;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (accumulate) return DGR_OK;
        return cudaMemsetAsync(out, 0, H * 4, s) == cudaSuccess ? DGR_OK : DGR_ERR_CUDA;
    }

    ColsumParams p{};
    p.x = static_cast<const char *>(x);
    p.stride_b = stride_b;
    p.stride_s = stride_s;
    p.S = static_cast<int32_t>(S);
    p.T = static_cast<int32_t>(T);
    p.H = static_cast<int32_t>(H);
    p.W = tile_rows;
    p.n_tiles = L.n_tiles;
    p.flat = (B == 1 || stride_b == S * stride_s) ? 1 : 0;
    const int vec = 16 / esize;
    const bool vec_ok = aligned(x, 16) && (H % vec) == 0 && (stride_s * esize) % 16 == 0 &&
                        (stride_b * esize) % 16 == 0;
    int VE = 1, rpt = 1, rpl = 0;
    colsum_geometry(p, H, tile_rows, esize, vec_ok, L.n_tiles, VE, rpt, rpl);
    p.FC = L.FC;
    p.n_fcb = L.n_fcb;
    p.batch = (kFolderSmemBytes / (2 * p.FC * 4)) & ~3;  // a multiple of 4: the chain reads 16-byte groups
    p.out = out;
    p.accumulate = accumulate ? 1 : 0;
    char *w = static_cast<char *>(ws);
    p.hdr = reinterpret_cast<WsHeader *>(w);
    p.counters = reinterpret_cast<int32_t *>(w + L.counters_off);
    p.slots = reinterpret_cast<float *>(w + L.slots_off);
    p.col_stride = L.col_stride;
    // producer scratch: TPC * RG * CB * VE floats must fit the launch's shared memory
    if (static_cast<size_t>(p.TPC) * p.RG * p.CB * VE * 4 > static_cast<size_t>(kFolderSmemBytes))
        return DGR_ERR_UNSUPPORTED;
    const bool warp_producers = p.stream_mode != 0;
    if (warp_producers) p.n_pcb = 1;
    const int64_t n_units = warp_producers ? L.n_tiles : (L.n_tiles + p.TPC - 1) / p.TPC * p.n_pcb;
    if (n_units > INT32_MAX) return DGR_ERR_UNSUPPORTED;
    p.n_units = static_cast<int32_t>(n_units);
    p.sched = sched_for(static_cast<uint32_t>(n_units));
    ColsumKernel k = nullptr;
    if (warp_producers && L.n_tiles <= kSmallTiles)
        k = dtype == DGR_DTYPE_BF16 ? small_kernel<DGR_DTYPE_BF16, 8>(rpl) : small_kernel<DGR_DTYPE_F32, 4>(rpl);
    else if (warp_producers)
        k = dtype == DGR_DTYPE_BF16 ? warp_kernel<DGR_DTYPE_BF16, 8>(rpl) : warp_kernel<DGR_DTYPE_F32, 4>(rpl);
    else if (dtype == DGR_DTYPE_BF16)
        k = VE == 8 ? cta_kernel<DGR_DTYPE_BF16, 8>(rpt) : cta_kernel<DGR_DTYPE_BF16, 1>(rpt);
    else
        k = VE == 4 ? cta_kernel<DGR_DTYPE_F32, 4>(rpt) : cta_kernel<DGR_DTYPE_F32, 1>(rpt);
    if (!k) return DGR_ERR_INVALID_ARG;
    int sms = 0, occ = 1;
    dgr_status st = usable_sms(&sms);
    if (st != DGR_OK) return st;
    const bool small = warp_producers && L.n_tiles <= kSmallTiles;
    const size_t smem = small ? 0 : (warp_producers ? kWarpSmemBytes : kFolderSmemBytes);
    const unsigned threads = small ? kSmallWarps * 32 : (warp_producers ? kWarpThreads : kThreads);
    if (warp_producers && !small &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kWarpSmemBytes) != cudaSuccess)
        return DGR_ERR_CUDA;
    if (!warp_producers && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, smem) != cudaSuccess)
        return DGR_ERR_CUDA;
    const ColsumPlan pl = colsum_plan(L.n_tiles, L.n_fcb, n_units, warp_producers, sms, occ, p.sched.cap);
    if (pl.prod_ctas + pl.fold_ctas > INT32_MAX) return DGR_ERR_UNSUPPORTED;
    if (pl.launches == 1) {
        p.fold_ctas = small ? 0 : pl.fold_ctas;
        k<<<static_cast<unsigned>(p.fold_ctas + pl.prod_ctas), threads, smem, s>>>(p);
        return launch_status();
    }
    p.fold_ctas = 0;  // producers only: every tile written and counted
    k<<<static_cast<unsigned>(pl.prod_ctas), threads, smem, s>>>(p);
    p.fold_ctas = pl.fold_ctas;  // then the folders, whose waits find every count complete
    k<<<static_cast<unsigned>(pl.fold_ctas), threads, smem, s>>>(p);
    return launch_status();
}

}  // namespace
}  // namespace dgr

extern "C" dgr_status dgr_ordered_colsum(const void *x, int32_t dtype, int64_t B, int64_t S, int64_t H,
                                         int64_t stride_b, int64_t stride_s, float *out,
                                         int32_t accumulate, int32_t tile_rows, void *ws, size_t ws_bytes,
                                         void *stream) {
    bool nothing = false;
    dgr_status st = colsum_args(x, dtype, B, S, H, stride_b, stride_s, out, tile_rows, nothing);
    if (st != DGR_OK || nothing) return st;
    const int64_t T = B * S;
    const Layout L = colsum_layout(T, H, tile_rows);
    if (T > 0) {
        if (!ws) return DGR_ERR_INVALID_ARG;
        if (ws_bytes < L.total) return DGR_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(ws, kAlign)) return DGR_ERR_MISALIGNED;
    }
    if ((st = colsum_input_checks(x, dtype, B, S, H, stride_b, stride_s, out)) != DGR_OK) return st;
    if (T > 0 && ranges_overlap(out, H * 4, ws, L.total)) return DGR_ERR_ALIAS;
    if ((st = check_device()) != DGR_OK) return st;
    return colsum_enqueue(x, dtype, B, S, H, stride_b, stride_s, out, accumulate, tile_rows, ws, stream);
}

extern "C" dgr_status dgr_diag_colsum_plan(int64_t T, int64_t H, int32_t tile_rows, int32_t dtype, int32_t vec_ok,
                                           int32_t sms, int32_t cta_occupancy, int32_t grid_cap, int32_t *plan) {
    if (!plan || T < 0 || T > INT32_MAX || H < 1 || H > 4096 || !is_pow2(tile_rows) || tile_rows > 4096 ||
        (dtype != DGR_DTYPE_BF16 && dtype != DGR_DTYPE_F32) || sms < 1 || cta_occupancy < 1 || grid_cap < 0)
        return DGR_ERR_INVALID_ARG;
    if (T == 0) {  // nothing is launched (out is written by a memset, or left)
        plan[0] = -1;
        plan[1] = plan[2] = plan[3] = 0;
        return DGR_OK;
    }
    const Layout L = colsum_layout(T, H, tile_rows);
    ColsumParams p{};
    int VE = 1, rpt = 1, rpl = 0;
    colsum_geometry(p, H, tile_rows, dtype == DGR_DTYPE_BF16 ? 2 : 4, vec_ok != 0, L.n_tiles, VE, rpt, rpl);
    const bool warp_producers = p.stream_mode != 0;
    const int64_t n_units = warp_producers ? L.n_tiles : (L.n_tiles + p.TPC - 1) / p.TPC * p.n_pcb;
    const ColsumPlan pl = colsum_plan(L.n_tiles, L.n_fcb, n_units, warp_producers, sms, cta_occupancy, grid_cap);
    plan[0] = pl.path;
    plan[1] = pl.launches;
    plan[2] = static_cast<int32_t>(pl.prod_ctas);
    plan[3] = pl.fold_ctas;
    return DGR_OK;
}

// ---------------------------------------------------------------------------
// Column sum without a caller workspace.
//
// For callers that cannot allocate device memory at the point where they need
// the reduction: code running inside another allocator's critical section,
// plugins handed only input and output pointers by a host framework that owns
// all device memory, or hot paths where a cudaMalloc would synchronise the
// device. Their scratch is this file-scope array instead (4 MiB, held on every
// GPU that loads the library until the process exits). The host cannot use
// the array's name as a device address (it is a host-side stand-in), so the
// first call on each device looks the address up with cudaGetSymbolAddress
// while that device is current and keeps it (only a lookup that succeeded is
// kept). A device-side error of a call is recorded in the array's first word,
// which dgr_colsum_noalloc_read_status() reads.
// ---------------------------------------------------------------------------
#include <atomic>
#include <mutex>

namespace dgr {
namespace {

constexpr size_t kStaticScratchBytes = DGR_COLSUM_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_colsum_scratch[kStaticScratchBytes];

// Device addresses of the array, one per device, set only by a lookup that
// succeeded (a failed one, e.g. during a stream capture, is tried again).
std::atomic<void *> g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

}  // namespace

dgr_status noalloc_scratch(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DGR_ERR_UNSUPPORTED;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (!p) {
            if (cudaGetSymbolAddress(&p, g_colsum_scratch) != cudaSuccess || !p) {
                cudaGetLastError();
                return DGR_ERR_CUDA;
            }
            g_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *ptr = p;
    return DGR_OK;
}

}  // namespace dgr

extern "C" dgr_status dgr_ordered_colsum_noalloc(const void *x, int32_t dtype, int64_t B, int64_t S, int64_t H,
                                                 int64_t stride_b, int64_t stride_s, float *out,
                                                 int32_t accumulate, int32_t tile_rows, void *stream) {
    // every argument is checked before the shared array is touched: a refused
    // call enqueues nothing
    bool nothing = false;
    dgr_status st = colsum_args(x, dtype, B, S, H, stride_b, stride_s, out, tile_rows, nothing);
    if (st != DGR_OK || nothing) return st;
    const int64_t T = B * S;
    const Layout L = colsum_layout(T, H, tile_rows);
    if (L.total > kStaticScratchBytes) return DGR_ERR_WORKSPACE_TOO_SMALL;
    if ((st = colsum_input_checks(x, dtype, B, S, H, stride_b, stride_s, out)) != DGR_OK) return st;
    if ((st = check_device()) != DGR_OK) return st;
    void *ws = nullptr;
    if ((st = noalloc_scratch(&ws)) != DGR_OK) return st;
    // The array keeps whatever the previous call (of any shape, or one that
    // ended in an error) left; the call's whole region starts at zero.
    if (T > 0 && cudaMemsetAsync(ws, 0, L.total, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DGR_ERR_CUDA;
    return colsum_enqueue(x, dtype, B, S, H, stride_b, stride_s, out, accumulate, tile_rows, ws, stream);
}

extern "C" dgr_status dgr_colsum_noalloc_read_status(int32_t clear, int32_t *status, void *stream) {
    if (!status) return DGR_ERR_INVALID_ARG;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    void *ws = nullptr;
    if ((st = noalloc_scratch(&ws)) != DGR_OK) return st;
    return dgr_read_device_status(ws, clear, status, stream);
}
