// Split-K grouped weight gradient accumulated into fp32 main_grad.
//
// FlashInfer PR #8602 (fuse the fp32 weight-gradient accumulate into
// main_grad) and follow-up #8924 ("Design and numerics"): out[e] gets
// G_e^T X_e added; the deterministic route computes dW in a fixed order and
// then RN32(out + dW); an empty group leaves out bitwise unchanged; the split
// tail was the only order-varying launch. Here the split order is fixed:
//   p_c = the chunk's G^T X on the tensor cores, chunks of 512 tokens from the
//         expert's first token, a fresh accumulator per chunk, K16 steps in
//         ascending token order;
//   dW  = fold_c p_c (ascending, in registers of the epilogue warps);
//   main_grad = RN(main_grad + dW), in the same kernel: the epilogue hands dW
//         to the bulk copy engine's tensor reduce-add, which adds it into
//         main_grad in L2 (one round-to-nearest add per element, subnormals
//         kept; each element has exactly this one writer, so no order is
//         involved).
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles (n x k) walked
// expert by expert; when the last wave of tiles would keep at most half the
// CTAs busy, its tiles run as halves of 128 k columns (MMA N = 128) instead,
// twice as many items of half the work (each output element is computed the
// same way by either MMA shape). Warp 0 issues TMA loads (64-token stages, 128-byte
// swizzle; G and X are MN-major as they lie in memory, so no transpose), warp
// 1 issues tcgen05.mma into one of two TMEM accumulators (256 columns each),
// warps 4-11 read the accumulator back, fold the chunks and finish the tile
// (the epilogue warpgroups hold the running fold, 128 fp32 per thread, so
// they take most of the registers; warps 2-3 idle) and issue the tile's
// reduce-adds through a 16 KB shared-memory box per column half.
// Rows of a stage past the expert's end are zeroed in shared memory before
// the MMA reads them (TMA fills rows past the tensor's end with zeros).
// Every wait is bounded; a timeout records DGR_ERR_TIMEOUT and aborts the
// CTA, which then waits (bounded again) for its own TMA copies in flight and
// for the completion of the MMAs it issued before it frees its TMEM.
#include <mutex>

#include <cudaTypedefs.h>

#include "tc_common.cuh"
#include "dgr_diag.h"

namespace dgr {
namespace {

using namespace tc;

constexpr int BM = 128;                 // n per tile (TMEM lanes)
constexpr int BN = 256;                 // k per tile (TMEM columns per accumulator)
constexpr int BK = 64;                  // tokens per pipeline stage
constexpr int kStages = 4;
constexpr int kChunk = 512;
constexpr int kEpiWarps = 8;
constexpr int kThreadsW = (4 + kEpiWarps) * 32;  // warpgroup 0: TMA, MMA, 2 idle; warpgroups 1-2: epilogue
// Register split: launched at 168 per thread (3 warps per SM sub-partition),
// warpgroup 0 gives back to 56 and the epilogue warpgroups take 224:
// 128 * 56 + 256 * 224 = 384 * 168.
constexpr int kRegsLow = 56;
constexpr int kRegsHigh = 224;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= 384 * 168, "register split exceeds the launch's registers");
constexpr uint32_t kBoxBytes = 64 * 128;                  // one 64 x 64 bf16 atom (128-byte swizzle)
constexpr uint32_t kStageA = 2 * kBoxBytes;               // 128 n x 64 tokens
constexpr uint32_t kStageB = 4 * kBoxBytes;               // 256 k x 64 tokens
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr uint32_t kLBO = kBoxBytes;                      // between 64-wide atoms along n / k
constexpr uint32_t kSBO = 1024;                           // between 8-token row groups
constexpr uint32_t kIdesc = idesc_bf16_mn(BM, BN);
constexpr uint32_t kIdescHalf = idesc_bf16_mn(BM, BN / 2);  // a half tile: 128 k columns
constexpr uint32_t kTmemCols = 2 * BN;

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t gsync[2];  // the four epilogue warps of a column half, per reduce-add box
    uint64_t dead;      // never arrived at: the diagnostic stall waits on it
    uint32_t tmem_base;
    int abort;
};
// per epilogue column half (four warps), one 128 x 32 fp32 box (16 KB,
// 1024-byte aligned) for the reduce-add of a 32-column slice of the tile's 128
// rows, in the 128-byte swizzle of the main_grad tensor map; warp q writes
// rows 32q .. 32q + 31
constexpr uint32_t kBoxM = 32 * 32 * 4;
constexpr uint32_t kXposeBytes = kEpiWarps * kBoxM;
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + kXposeBytes + sizeof(Ctl);

struct WgradParams {
    const int64_t *offs;
    int32_t E, N, K;
    int32_t n_blk, k_blk, n_tiles;
    float *main_grad;
    WsHeader *hdr;
    // Work items: tiles below n_split whole, the rest as two halves of 128 k
    // columns each (items n_split + 2j and + 2j + 1), so that a last wave that
    // would leave more than half the CTAs idle is spread over twice as many.
    int32_t n_split, n_items;
    Sched sched;  // the order in which the CTAs walk the items
    // Diagnostic stall (dgr_diag_wgrad_stall; 0 in every product call): CTA 0's
    // role stall_role (1 TMA producer, 2 MMA issuer, 3 epilogue warp 4) waits on
    // a barrier nobody arrives at, at its stall_after-th stage (roles 1, 2) or
    // tile end (role 3), until stall_ns runs out; the CTA then aborts like on
    // any other timeout.
    int32_t stall_role, stall_after;
    uint64_t stall_ns;
};

// The diagnostic stall of role r at count n: false once its wait ran out.
__device__ __forceinline__ bool stall_point(const WgradParams &p, Ctl *ctl, volatile int *abort_flag, int r, int n) {
    if (p.stall_role != r || n != p.stall_after || blockIdx.x != 0) return true;
    return mbar_wait(&ctl->dead, 0, abort_flag, p.hdr, 14 + r, p.stall_ns);
}

// main_grad[y .. y + 127][x .. x + 31] += the box at src (bulk async group).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the thread's committed bulk operations have read their shared memory
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and are complete
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t a, float x, float y, float z, float w) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w) : "memory");
}

// The k-th of this CTA's n_my work items: items blockIdx, blockIdx + G, ...
// (G CTAs), except that an odd CTA whose last item is a half tile takes that
// half first. Every tile has the same token count, so the CTAs would otherwise
// reach their tile ends, and send their main_grad reduce-adds, all at once;
// half of them then run about half a tile out of phase instead (424 -> 419 us
// a call, the same bits: the items and their arithmetic are unchanged).
__device__ __forceinline__ int my_item(const WgradParams &p, int k, int n_my) {
    const int b = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const int last = b + (n_my - 1) * G;
    if ((b & 1) && n_my > 1 && last >= p.n_split) return k == 0 ? last : b + (k - 1) * G;
    return b + k * G;
}
// how many items this CTA takes
__device__ __forceinline__ int my_items(const WgradParams &p) {
    const int b = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    return b < p.n_items ? (p.n_items - b + G - 1) / G : 0;
}

// item -> tile, and its half (-1: the whole tile)
__device__ __forceinline__ int item_tile(const WgradParams &p, int item, int &half) {
    if (item < p.n_split) {
        half = -1;
        return item;
    }
    const int j = item - p.n_split;
    half = j & 1;
    return p.n_split + (j >> 1);
}

__device__ __forceinline__ void tile_coords(const WgradParams &p, int tau, int &e, int &nb, int &kb) {
    const int per = p.n_blk * p.k_blk;
    e = tau / per;
    const int r = tau - e * per;
    nb = r / p.k_blk;
    kb = r - nb * p.k_blk;
}

__device__ __forceinline__ void expert_range(const WgradParams &p, int e, int32_t &t_beg, int32_t &te) {
    const int64_t a = p.offs[e];
    const int64_t b = p.offs[e + 1];
    t_beg = static_cast<int32_t>(a);
    te = static_cast<int32_t>(b > a ? b - a : 0);
}

__global__ void __launch_bounds__(kThreadsW, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmX,
                 const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmM,
                 const WgradParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xbox = smem + kStages * kStageBytes;
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + kStages * kStageBytes + kXposeBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int *abort_flag = &ctl->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], kEpiWarps);
            mbar_init(&ctl->gsync[b], 4);
        }
        mbar_init(&ctl->dead, 1);
        ctl->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmX2);
        prefetch_tmap(&tmM);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp < 4) setmaxnreg_dec<kRegsLow>();

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool armed[kStages] = {};
            uint32_t armed_phase[kStages] = {};
            bool ok = true;
            int n_stage = 0;
            for (int k = 0, n_my = my_items(p); ok && k < n_my; ++k) {
                const int tau = my_item(p, k, n_my);
                int e, nb, kb;
                int half;
                tile_coords(p, item_tile(p, static_cast<int>(sched_item(p.sched, tau)), half), e, nb, kb);
                int32_t t_beg, te;
                expert_range(p, e, t_beg, te);
                for (int32_t c0 = 0; ok && c0 < te; c0 += kChunk) {
                    const int32_t vc = min(kChunk, te - c0);
                    for (int32_t s0 = 0; s0 < vc; s0 += BK) {
                        if (!stall_point(p, ctl, abort_flag, 1, n_stage++) ||
                            !mbar_wait(&ctl->empty[stage], phase ^ 1, abort_flag, p.hdr, 10)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sA = smem + stage * kStageBytes;
                        uint8_t *sB = sA + kStageA;
                        const int32_t t = t_beg + c0 + s0;
                        mbar_arrive_expect_tx(&ctl->full[stage], half < 0 ? kStageBytes : kStageA + 2 * kBoxBytes);
                        armed[stage] = true;
                        armed_phase[stage] = phase;
                        // G: 2 column blocks of 64, X: 4, one copy each
                        tma_load_3d(sA, &tmG, &ctl->full[stage], 0, t, nb * (BM / 64));
                        if (half < 0) tma_load_3d(sB, &tmX, &ctl->full[stage], 0, t, kb * (BN / 64));
                        else tma_load_3d(sB, &tmX2, &ctl->full[stage], 0, t, kb * (BN / 64) + 2 * half);
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                }
            }
            if (!ok) {  // aborted: let our copies in flight land (bounded) before the CTA exits
                int dummy = 0;
                for (int s = 0; s < kStages; ++s)
                    if (armed[s]) mbar_wait(&ctl->full[s], armed_phase[s], &dummy, nullptr, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        uint32_t stage = 0, phase = 0, g = 0;
        uint32_t last_stage = 0, last_phase = 0;  // the latest stage-release commit
        bool committed = false, ok = true;
        int n_stage = 0;
        for (int k = 0, n_my = my_items(p); ok && k < n_my; ++k) {
            const int tau = my_item(p, k, n_my);
            int e, nb, kb;
            int half;
            tile_coords(p, item_tile(p, static_cast<int>(sched_item(p.sched, tau)), half), e, nb, kb);
            int32_t t_beg, te;
            expert_range(p, e, t_beg, te);
            for (int32_t c0 = 0; ok && c0 < te; c0 += kChunk, ++g) {
                const int32_t vc = min(kChunk, te - c0);
                const uint32_t buf = g & 1, tph = (g >> 1) & 1;
                if (!mbar_wait(&ctl->tempty[buf], tph ^ 1, abort_flag, p.hdr, 11)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * BN;
                for (int32_t s0 = 0; s0 < vc; s0 += BK) {
                    if (!stall_point(p, ctl, abort_flag, 2, n_stage++) ||
                        !mbar_wait(&ctl->full[stage], phase, abort_flag, p.hdr, 12)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint8_t *sA = smem + stage * kStageBytes;
                    uint8_t *sB = sA + kStageA;
                    const int vst = min(BK, vc - s0);
                    const int nk = (vst + 15) / 16;
                    if (vst & 15) {
                        // tokens [vst, 16*nk) of this stage belong to the next
                        // expert (or lie past the tensor): zero them in A and B
                        const int rows = 16 * nk - vst;
                        for (int q = lane; q < 6 * rows * 8; q += 32) {
                            const int box = q / (rows * 8);
                            const int rr = (q / 8) % rows + vst;
                            const int ch = q % 8;
                            uint8_t *b = (box < 2 ? sA + box * kBoxBytes : sB + (box - 2) * kBoxBytes);
                            *reinterpret_cast<uint4 *>(b + rr * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    if (lane == 0) {
                        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
                        if (nk == 4) {
                            // a whole stage: the four MMAs issued back to back with
                            // their descriptors ready (scalar work between
                            // consecutive MMAs keeps the tensor pipe from
                            // overlapping them: measured 2.3x slower per MMA)
                            uint64_t ad[4], bd[4];
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                ad[kk] = smem_desc_sw128(a0 + kk * 2048, kLBO, kSBO);
                                bd[kk] = smem_desc_sw128(b0 + kk * 2048, kLBO, kSBO);
                            }
                            const uint32_t acc0 = s0 > 0 ? 1u : 0u;
                            const uint32_t idesc = half < 0 ? kIdesc : kIdescHalf;
                            mma_bf16(d_tmem, ad[0], bd[0], idesc, acc0);
                            mma_bf16(d_tmem, ad[1], bd[1], idesc, 1u);
                            mma_bf16(d_tmem, ad[2], bd[2], idesc, 1u);
                            mma_bf16(d_tmem, ad[3], bd[3], idesc, 1u);
                        } else {
                            for (int kk = 0; kk < nk; ++kk) {
                                const uint64_t ad = smem_desc_sw128(a0 + kk * 2048, kLBO, kSBO);
                                const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, kLBO, kSBO);
                                mma_bf16(d_tmem, ad, bd, half < 0 ? kIdesc : kIdescHalf, (s0 > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                        mma_commit(&ctl->empty[stage]);
                    }
                    __syncwarp();
                    committed = true;
                    last_stage = stage;
                    last_phase = phase;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (lane == 0) mma_commit(&ctl->tfull[buf]);
                __syncwarp();
            }
        }
        if (!ok && committed) {
            // aborted: the tensor pipe may still be running MMAs issued here;
            // the latest commit completes once all of them are done (bounded),
            // and only then may the CTA free its TMEM and exit
            int dummy = 0;
            mbar_wait(&ctl->empty[last_stage], last_phase, &dummy, nullptr, kWaitLimitNs);
        }
    } else if (warp >= 4) {
        // ---------------- epilogue: fold chunks, add into main_grad ----------------
        setmaxnreg_inc<kRegsHigh>();
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int h = (warp - 4) >> 2;          // column half of the tile
        uint32_t g = 0, gph = 0;
        bool ok = true;
        int n_end = 0;
        // main_grad += dW, a 32-column slice at a time (send): the four warps of
        // the column half write their rows into the half's box (row i of a warp
        // from lane i, as TMEM gives them, in the map's 128-byte swizzle: 16-byte
        // chunk c of a row at chunk c ^ (row % 8), so the 32 lanes' stores spread
        // over the banks), and one tensor reduce-add, issued by warp q = 0, sends
        // the 128 x 32 box to main_grad; the box is written again once the engine
        // has read it. The four warps meet on an mbarrier (bounded waits) before
        // writing the box and before it is sent. The SM never reads main_grad:
        // the add happens in L2 (442 us a call with the read-modify-write in the
        // epilogue warps, through a transpose tile, after an L2 prefetch of the
        // tile's main_grad; 423 us with a reduce-add of a 32 x 32 box per warp;
        // 414.5 against 416.8 us with one per column half). A tile's last slice
        // goes out one chunk later, after the next tile's first accumulator is
        // read, so that less of every SM's update traffic falls on the moment
        // all CTAs reach their tile ends (423.7-424.0 against 426.5-428.7 us;
        // deferring two slices needs more registers than the warps have). The
        // same bits every way.
        float F[4][32];
        float Fd[32];           // the last slice of the previous tile, sent one chunk later
        bool have_def = false;
        int32_t def_rowg = 0, def_col = 0;
        const bool issuer = q == 0 && lane == 0;
        const uint32_t gbox = smem_u32(xbox) + h * (4 * kBoxM);
        const uint32_t xs = gbox + q * kBoxM;
        auto group_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->gsync[h]);
            const bool r = mbar_wait(&ctl->gsync[h], gph, abort_flag, p.hdr, 14);
            gph ^= 1;
            return r;
        };
        // one 32-column slice of the column half's 128 rows to main_grad
        auto send = [&](const float (&v)[32], int32_t col, int32_t rowg) -> bool {
            if (issuer) bulk_wait_read0();
            if (!group_sync()) return false;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(xs + lane * 128 + 16 * (c ^ (lane & 7)), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            fence_proxy_async_smem();
            if (!group_sync()) return false;
            if (issuer) {
                tma_reduce_add_2d(&tmM, gbox, col, rowg);
                bulk_commit();
            }
            return true;
        };
        for (int k = 0, n_my = my_items(p); ok && k < n_my; ++k) {
            const int tau = my_item(p, k, n_my);
            int e, nb, kb;
            int half;
            tile_coords(p, item_tile(p, static_cast<int>(sched_item(p.sched, tau)), half), e, nb, kb);
            int32_t t_beg, te;
            expert_range(p, e, t_beg, te);
            if (te == 0) continue;  // empty expert: main_grad untouched
            const bool active = half < 0 || h == 0;
            const int coff = half < 0 ? 128 * h : 128 * half;
            for (int32_t c0 = 0; c0 < te; c0 += kChunk, ++g) {
                const uint32_t buf = g & 1, tph = (g >> 1) & 1;
                if (!mbar_wait(&ctl->tfull[buf], tph, abort_flag, p.hdr, 13)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t base = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * BN + (half < 0 ? 128 * h : 0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (!active) break;
                    uint32_t r[32];
                    tmem_ld32(base + 32 * j, r);
                    tmem_wait_ld(r);
                    if (c0 == 0) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) F[j][i] = __uint_as_float(r[i]);
                    } else {
                        // packed pairs: the same bits as 32 scalar adds, half the issue
                        // slots (434.2 -> 426.3 us a call, alternating on one box)
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 d = add2(make_float2(F[j][i], F[j][i + 1]),
                                                  make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])));
                            F[j][i] = d.x;
                            F[j][i + 1] = d.y;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
                if (c0 == 0 && have_def) {  // the previous tile's last slice, a chunk after its others
                    if (!send(Fd, def_col, def_rowg)) {
                        ok = false;
                        break;
                    }
                    have_def = false;
                }
            }
            if (!ok) break;
            if (!active) continue;
            if (warp == 4 && !stall_point(p, ctl, abort_flag, 3, n_end)) {
                ok = false;
                break;
            }
            ++n_end;
            const int32_t rowg = e * p.N + nb * BM;
            const int32_t col0 = kb * BN + coff;
            if (!send(F[0], col0, rowg) || !send(F[1], col0 + 32, rowg) || !send(F[2], col0 + 64, rowg)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) Fd[i] = F[3][i];
            have_def = true;
            def_rowg = rowg;
            def_col = col0 + 96;
        }
        if (ok && have_def) send(Fd, def_col, def_rowg);
    }
    if (warp >= 4 && lane == 0) bulk_wait0();  // the warp's last reduce-adds are done
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// One K16 tensor-core step per CTA on caller data: D = [C +] A B, with A
// [128 x 16] and B [16 x 256] bf16 placed in the same MN-major 128-byte
// swizzle layout and descriptors as the wgrad kernel's stages. Used to check
// the oracle's model of the step and the layout itself.
// The probe holds a large allocation so that its descriptors can only ever
// address shared memory the CTA owns.
constexpr size_t kProbeSmem = 200 * 1024;

__global__ void __launch_bounds__(128, 1)
    tc_probe_kernel(const uint16_t *A, const uint16_t *B, const float *C, float *D, int accumulate, WsHeader *hdr) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStageA;
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + kStageBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t prob = blockIdx.x;
    A += prob * 128 * 16;
    B += prob * 16 * 256;
    C += prob * 128 * 256;
    D += prob * 128 * 256;
    for (int i = tid; i < static_cast<int>(kStageBytes / 16); i += 128)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    for (int i = tid; i < 128 * 16; i += 128) {
        const int m = i / 16, k = i % 16;
        *reinterpret_cast<uint16_t *>(sA + sw128_mn_offset(m, k, kLBO)) = A[i];
    }
    for (int i = tid; i < 16 * 256; i += 128) {
        const int k = i / 256, n = i % 256;
        *reinterpret_cast<uint16_t *>(sB + sw128_mn_offset(n, k, kLBO)) = B[i];
    }
    fence_proxy_async_smem();
    if (tid == 0) {
        mbar_init(&ctl->full[0], 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&ctl->tmem_base, BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    const int row = 32 * warp + lane;
#pragma unroll 1
    for (int j = 0; j < BN / 32; ++j) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(C[row * 256 + 32 * j + i]);
        tmem_st32(lane_base + 32 * j, r);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        mma_bf16(tmem, smem_desc_sw128(smem_u32(sA), kLBO, kSBO), smem_desc_sw128(smem_u32(sB), kLBO, kSBO), kIdesc,
                 accumulate ? 1u : 0u);
        mma_commit(&ctl->full[0]);
    }
    __syncwarp();
    const bool ok = mbar_wait(&ctl->full[0], 0, &ctl->abort, hdr, 20);
    tc_fence_after();
    if (ok) {
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
            uint32_t r[32];
            tmem_ld32(lane_base + 32 * j, r);
            tmem_wait_ld(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) D[row * 256 + 32 * j + i] = __uint_as_float(r[i]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, BN);
    }
}

// ---- host ---------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

dgr_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000 *fn) {
    std::call_once(g_encode_once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    if (!g_encode) return DGR_ERR_CUDA;
    *fn = g_encode;
    return DGR_OK;
}

// Tensor map over a row-major bf16 [rows, cols] matrix (cols a multiple of 64)
// viewed as {64 columns, rows, cols / 64 blocks}: a box of 64 rows and
// `blocks` column blocks lands as `blocks` consecutive 64 x 64 atoms (8 KB
// each), 128-byte swizzle, zero fill past the last row.
dgr_status make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t blocks) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    dgr_status st = encode_fn(&enc);
    if (st != DGR_OK) return st;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols * 2), 128};
    const cuuint32_t box[3] = {64, 64, blocks};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DGR_OK : DGR_ERR_CUDA;
}

// Tensor map over main_grad as fp32 [rows, cols] row-major: a box of 128 rows x
// 32 columns (128 bytes a row), 128-byte swizzle.
dgr_status make_mg_map(CUtensorMap *m, void *base, int64_t rows, int64_t cols) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    dgr_status st = encode_fn(&enc);
    if (st != DGR_OK) return st;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 4)};
    const cuuint32_t box[2] = {32, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DGR_OK : DGR_ERR_CUDA;
}

std::once_flag g_attr_once[64];
cudaError_t g_attr_err[64];

dgr_status set_smem_attrs() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DGR_ERR_CUDA;
    std::call_once(g_attr_once[dev], [dev] {
        cudaError_t e = cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tc_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kProbeSmem));
        g_attr_err[dev] = e;
    });
    return g_attr_err[dev] == cudaSuccess ? DGR_OK : DGR_ERR_CUDA;
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" size_t dgr_wgrad_workspace_bytes(int32_t E, int64_t N, int64_t K) {
    (void)E;
    (void)N;
    (void)K;
    return sizeof(WsHeader);
}

namespace dgr {
namespace {

dgr_status wgrad_call(const void *G, const void *X, const int64_t *d_offs, int32_t E, int64_t T_total, int64_t N,
                      int64_t K, float *main_grad, int32_t chunk_tokens, void *ws, size_t ws_bytes, void *stream,
                      int32_t stall_role, int32_t stall_after, uint64_t stall_ns) {
    if (E < 1 || T_total < 0 || N <= 0 || K <= 0 || chunk_tokens != kChunk) return DGR_ERR_INVALID_ARG;
    if (N % BM != 0 || K % BN != 0 || T_total >= INT32_MAX || N > (1 << 20) || K > (1 << 20) ||
        static_cast<int64_t>(E) * N > INT32_MAX)
        return DGR_ERR_UNSUPPORTED;
    if (!main_grad || !d_offs || !ws || (T_total > 0 && (!G || !X))) return DGR_ERR_INVALID_ARG;
    if (ws_bytes < sizeof(WsHeader)) return DGR_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(G, 16) || !aligned(X, 16) || !aligned(main_grad, 32) || !aligned(d_offs, 8) ||
        !aligned(ws, kAlign))
        return DGR_ERR_MISALIGNED;
    const size_t mg_bytes = static_cast<size_t>(E) * N * K * 4;
    if (ranges_overlap(main_grad, mg_bytes, G, T_total * N * 2) ||
        ranges_overlap(main_grad, mg_bytes, X, T_total * K * 2) ||
        ranges_overlap(main_grad, mg_bytes, d_offs, (E + 1) * 8) || ranges_overlap(main_grad, mg_bytes, ws, ws_bytes))
        return DGR_ERR_ALIAS;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    if (T_total == 0) return DGR_OK;
    st = set_smem_attrs();
    if (st != DGR_OK) return st;
    CUtensorMap mG, mX, mX2;
    if ((st = make_map(&mG, G, T_total, N, BM / 64)) != DGR_OK) return st;
    if ((st = make_map(&mX, X, T_total, K, BN / 64)) != DGR_OK) return st;
    if ((st = make_map(&mX2, X, T_total, K, BN / 128)) != DGR_OK) return st;
    CUtensorMap mM;  // main_grad as [E * N, K]: the row coordinate fits 32 bits
    if ((st = make_mg_map(&mM, main_grad, static_cast<int64_t>(E) * N, K)) != DGR_OK) return st;
    WgradParams p{};
    p.offs = d_offs;
    p.E = E;
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.n_blk = static_cast<int32_t>(N / BM);
    p.k_blk = static_cast<int32_t>(K / BN);
    const int64_t n_tiles = static_cast<int64_t>(E) * p.n_blk * p.k_blk;
    if (n_tiles > INT32_MAX) return DGR_ERR_UNSUPPORTED;
    p.n_tiles = static_cast<int32_t>(n_tiles);
    p.main_grad = main_grad;
    p.hdr = static_cast<WsHeader *>(ws);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DGR_ERR_CUDA;
    // a last wave filling at most half the CTAs runs as half tiles instead
    const int64_t G0 = n_tiles < sms ? n_tiles : sms;
    const int64_t rem = n_tiles % G0;
    p.n_split = static_cast<int32_t>(rem > 0 && 2 * rem <= G0 ? n_tiles - rem : n_tiles);
    const int64_t n_items = p.n_split + 2 * (n_tiles - p.n_split);
    if (n_items > INT32_MAX) return DGR_ERR_UNSUPPORTED;
    p.n_items = static_cast<int32_t>(n_items);
    p.sched = sched_for(static_cast<uint32_t>(n_items));
    p.stall_role = stall_role;
    p.stall_after = stall_after;
    p.stall_ns = stall_ns;
    const unsigned grid = sched_grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
    wgrad_kernel<<<grid, kThreadsW, kSmemBytes, static_cast<cudaStream_t>(stream)>>>(mG, mX, mX2, mM, p);
    return launch_status();
}

}  // namespace
}  // namespace dgr

extern "C" dgr_status dgr_grouped_wgrad_accumulate(const void *G, const void *X, const int64_t *d_offs, int32_t E,
                                                   int64_t T_total, int64_t N, int64_t K, float *main_grad,
                                                   int32_t chunk_tokens, void *ws, size_t ws_bytes, void *stream) {
    return wgrad_call(G, X, d_offs, E, T_total, N, K, main_grad, chunk_tokens, ws, ws_bytes, stream, 0, 0, 0);
}

extern "C" dgr_status dgr_diag_wgrad_stall(const void *G, const void *X, const int64_t *d_offs, int32_t E,
                                           int64_t T_total, int64_t N, int64_t K, float *main_grad, void *ws,
                                           size_t ws_bytes, int32_t role, int32_t after, int32_t limit_us,
                                           void *stream) {
    if (role < 1 || role > 3 || after < 0 || limit_us < 1 || limit_us > 1000000) return DGR_ERR_INVALID_ARG;
    return wgrad_call(G, X, d_offs, E, T_total, N, K, main_grad, kChunk, ws, ws_bytes, stream, role, after,
                      static_cast<uint64_t>(limit_us) * 1000ull);
}

extern "C" dgr_status dgr_tc_probe_k16(const uint16_t *A, const uint16_t *B, const float *C, float *D, int32_t n_prob,
                                       int32_t accumulate, void *ws, size_t ws_bytes, void *stream) {
    if (n_prob < 0 || !A || !B || !C || !D || !ws) return DGR_ERR_INVALID_ARG;
    if (ws_bytes < sizeof(WsHeader)) return DGR_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(A, 2) || !aligned(B, 2) || !aligned(C, 4) || !aligned(D, 4) || !aligned(ws, kAlign))
        return DGR_ERR_MISALIGNED;
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    if (n_prob == 0) return DGR_OK;
    st = set_smem_attrs();
    if (st != DGR_OK) return st;
    tc_probe_kernel<<<n_prob, 128, kProbeSmem, static_cast<cudaStream_t>(stream)>>>(
        A, B, C, D, accumulate, static_cast<WsHeader *>(ws));
    return launch_status();
}
