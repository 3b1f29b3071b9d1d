// dprob fused into its grouped dsReLU GEMM:
//   C = A_e B_e on the tensor cores (K16 steps ascending from a fresh
//   accumulator), leaf[m][n] = RN(fp32(dY[m][n]) * RN(relu(C[m][n])^2)),
//   dprob[m] = fold over N-tiles of 128 of pw_128(leaves), written or added.
//
// cuDNN-frontend PR #521 ("grouped gemm dsrelu deterministic dprob"): the
// backward kernel recomputes the grouped GEMM and reuses relu(C)^2 for dprob;
// determinism comes from one partial per (token, N-tile) with a single writer
// and a fixed-order reduction of the partials, accumulated into dprob. The
// GEMM output itself is never written: only its dprob partials leave the chip.
//
// Two launches:
//   gemm - persistent, one CTA per SM, 12 warps. Tiles are (expert, 128-row
//          block counted from the expert's first row, 256-column block),
//          expert by expert. Warp 0 loads 64-deep k stages by TMA (A [T, K]
//          K-major: one 128 x 64 atom; B_e [K, N] N-major: four 64 x 64
//          atoms in one copy; 128-byte swizzle, 4 stages); warp 1 issues tcgen05.mma (M 128,
//          N 256, K 16, bf16 in, fp32 in TMEM) over all of K into one of two
//          TMEM accumulators; warps 4-11 (lane quarter q, column half h) read
//          their row's 128 columns, form the leaves with the row of dY (its
//          loads issued before the accumulator is ready), sum them by the tile
//          tree in registers and store one partial per (row, N-tile).
//   fold - one thread per token, in plain stream order after the GEMM: its
//          N-tile partials folded in order into dprob. (Launched as a
//          programmatic dependent of the GEMM, with the GEMM releasing it at
//          its start, the pair took 266 us a call against 215 us this way.)
// Every wait is bounded; no floating-point value depends on timing. A timeout
// aborts the CTA, which then waits (bounded again) for its own TMA copies in
// flight and for the completion of the MMAs it issued before it frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_common.cuh"

namespace dgr {
namespace {

using namespace tc;

constexpr int BM = 128;  // rows of a tile (TMEM lanes)
constexpr int BN = 256;  // columns of a tile (TMEM columns per accumulator)
constexpr int BK = 64;   // k per stage (one 64-column block of A)
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (4 + kEpiWarps) * 32;
constexpr int kMaxExperts = 1024;
constexpr int kRegsLow = 56;
constexpr int kRegsHigh = 224;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= 384 * 168, "register split exceeds the launch's registers");
constexpr uint32_t kBoxA = BM * 128;            // 128 rows x 64 k (128 bytes a row)
constexpr uint32_t kBoxB = 64 * 128;            // one atom of B: 64 k rows x 64 n
static_assert(BK == 64, "a stage of A is one 64-column block of the map");
constexpr uint32_t kStageA = kBoxA;
constexpr uint32_t kStageB = 4 * kBoxB;         // 64 k x 256 n
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr uint32_t kSBO = 1024;                 // between 8-row groups
constexpr uint32_t kLboA = 16;                  // K-major, 128-byte swizzle: one atom spans the K16 step
constexpr uint32_t kLboB = kBoxB;               // N-major: between 64-wide atoms along n
// tcgen05 instruction descriptor: fp32 D, bf16 A and B, A K-major, B N-major
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                            (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
constexpr uint32_t kTmemCols = 2 * BN;

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t dead;  // never arrived at: the diagnostic stall waits on it
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + sizeof(Ctl);


struct DsParams {
    const int64_t *offs;
    int32_t E, T, K, N;
    int32_t nbs;          // 256-column blocks
    const uint16_t *dY;   // [T, N]
    float *slots;         // [T, N / 128]
    float *dprob;         // [T]
    int32_t accumulate;
    WsHeader *hdr;
    Sched sched;          // the setting; bound to the tile count on the device
    // Diagnostic stall (dgr_diag_dsrelu_stall; 0 in every product call): CTA 0's
    // role stall_role (1 TMA producer, 2 MMA issuer, 3 epilogue warp 4) waits on
    // a barrier nobody arrives at before its stall_after-th stage (roles 1, 2)
    // or accumulator (role 3), until stall_ns runs out, then aborts the CTA.
    int32_t stall_role, stall_after;
    uint64_t stall_ns;
};

// The diagnostic stall of role r at count n: false once its wait ran out.
__device__ __forceinline__ bool stall_point(const DsParams &p, Ctl *ctl, volatile int *abort_flag, int r, int64_t n) {
    if (p.stall_role != r || n != p.stall_after || blockIdx.x != 0) return true;
    return mbar_wait(&ctl->dead, 0, abort_flag, p.hdr, 40 + r, p.stall_ns);
}


// mb_base[e] = first m-block of expert e (mb_base[E] = all m-blocks), by the
// whole block; false when the offsets break the contract.
__device__ bool mblock_bases(const DsParams &p, int32_t *mb_base, int32_t *wsum, int32_t *bad) {
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, nt = blockDim.x, nw = nt >> 5;
    if (tid == 0) *bad = 0;
    __syncthreads();
    int32_t run = 0;
    for (int e0 = 0; e0 < p.E; e0 += nt) {
        const int e = e0 + tid;
        int32_t c = 0;
        if (e < p.E) {
            const int64_t a = p.offs[e], b = p.offs[e + 1];
            if (b < a || (e == 0 && a != 0) || (e == p.E - 1 && b != p.T)) *bad = 1;
            else c = static_cast<int32_t>((b - a + BM - 1) / BM);
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
        if (e < p.E) mb_base[e] = before + incl - c;
        for (int v = 0; v < nw; ++v) run += wsum[v];
        __syncthreads();
    }
    if (tid == 0) mb_base[p.E] = run;
    __syncthreads();
    return *bad == 0;
}

// tile tau -> expert, m-block within the expert, n-block
__device__ __forceinline__ void tile_of(const DsParams &p, const int32_t *mb_base, int64_t tau, int &e, int &mb,
                                        int &nb) {
    const int32_t gmb = static_cast<int32_t>(tau / p.nbs);
    nb = static_cast<int>(tau - static_cast<int64_t>(gmb) * p.nbs);
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mb_base[mid] <= gmb) lo = mid;
        else hi = mid - 1;
    }
    e = lo;
    mb = gmb - mb_base[lo];
}

__global__ void __launch_bounds__(kThreads, 1)
    dsrelu_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const DsParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + kStages * kStageBytes);
    __shared__ int32_t mb_base[kMaxExperts + 1];
    __shared__ int32_t wsum[kThreads / 32];
    __shared__ int32_t bad;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int *abort_flag = &ctl->abort;

    if (!mblock_bases(p, mb_base, wsum, &bad)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(p.hdr, DGR_ERR_INVALID_ARG, 30);
        return;
    }
    const int64_t n_tiles = static_cast<int64_t>(mb_base[p.E]) * p.nbs;
    const Sched sched = sched_over(p.sched, static_cast<uint32_t>(n_tiles));  // the tile count is known here only
    const int n_k = p.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], kEpiWarps);
        }
        mbar_init(&ctl->dead, 1);
        ctl->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
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
            int64_t n_stage = 0;
            for (int64_t tau = blockIdx.x; ok && tau < n_tiles; tau += gridDim.x) {
                int e, mb, nb;
                tile_of(p, mb_base, sched_item(sched, static_cast<uint32_t>(tau)), e, mb, nb);
                const int32_t row0 = static_cast<int32_t>(p.offs[e]) + mb * BM;
                for (int kb = 0; kb < n_k; ++kb) {
                    if (!stall_point(p, ctl, abort_flag, 1, n_stage++) ||
                        !mbar_wait(&ctl->empty[stage], phase ^ 1, abort_flag, p.hdr, 31)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sA = smem + stage * kStageBytes;
                    uint8_t *sB = sA + kStageA;
                    mbar_arrive_expect_tx(&ctl->full[stage], kStageBytes);
                    armed[stage] = true;
                    armed_phase[stage] = phase;
                    // A: one 64-column block of 128 rows; B: 4 blocks of 64 rows
                    tma_load_3d(sA, &tmA, &ctl->full[stage], 0, row0, kb);
                    tma_load_3d(sB, &tmB, &ctl->full[stage], 0, e * p.K + kb * BK, nb * (BN / 64));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
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
        int64_t n_stage = 0;
        for (int64_t tau = blockIdx.x; ok && tau < n_tiles; tau += gridDim.x, ++g) {
            const uint32_t buf = g & 1, tph = (g >> 1) & 1;
            if (!mbar_wait(&ctl->tempty[buf], tph ^ 1, abort_flag, p.hdr, 32)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + buf * BN;
            for (int kb = 0; kb < n_k; ++kb) {
                if (!stall_point(p, ctl, abort_flag, 2, n_stage++) ||
                    !mbar_wait(&ctl->full[stage], phase, abort_flag, p.hdr, 33)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a0 = smem_u32(smem + stage * kStageBytes), b0 = a0 + kStageA;
                    // the stage's four K16 steps back to back, descriptors ready
                    uint64_t ad[4], bd[4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        ad[kk] = smem_desc_sw128(a0 + kk * 32, kLboA, kSBO);
                        bd[kk] = smem_desc_sw128(b0 + kk * 2048, kLboB, kSBO);
                    }
                    mma_bf16(d_tmem, ad[0], bd[0], kIdesc, kb > 0 ? 1u : 0u);
                    mma_bf16(d_tmem, ad[1], bd[1], kIdesc, 1u);
                    mma_bf16(d_tmem, ad[2], bd[2], kIdesc, 1u);
                    mma_bf16(d_tmem, ad[3], bd[3], kIdesc, 1u);
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
        if (!ok && committed) {
            // aborted: wait (bounded) until the MMAs issued here are done, as
            // their latest commit says, before the CTA frees its TMEM and exits
            int dummy = 0;
            mbar_wait(&ctl->empty[last_stage], last_phase, &dummy, nullptr, kWaitLimitNs);
        }
    } else if (warp >= 4) {
        // ---------------- epilogue: leaves, tile trees, partials ----------------
        setmaxnreg_inc<kRegsHigh>();
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int h = (warp - 4) >> 2;    // N-tile (128 columns) within the 256-column block
        const int n_ntiles = p.N / 128;
        uint32_t g = 0;
        bool ok = true;
        for (int64_t tau = blockIdx.x; ok && tau < n_tiles; tau += gridDim.x, ++g) {
            int e, mb, nb;
            tile_of(p, mb_base, sched_item(sched, static_cast<uint32_t>(tau)), e, mb, nb);
            const int64_t row = p.offs[e] + static_cast<int64_t>(mb) * BM + 32 * q + lane;
            const bool mine = row < p.offs[e + 1];  // past the expert's end: not this expert's row
            // the row's 128 dY values, in flight while the accumulator fills
            const int col0 = nb * BN + 128 * h;
            uint4 dy[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                dy[i] = make_uint4(0u, 0u, 0u, 0u);
                ldg_nc_v4u_if(dy[i], p.dY + row * p.N + col0 + 8 * i, mine);
            }
            const uint32_t buf = g & 1, tph = (g >> 1) & 1;
            if ((warp == 4 && !stall_point(p, ctl, abort_flag, 3, static_cast<int64_t>(g))) ||
                !mbar_wait(&ctl->tfull[buf], tph, abort_flag, p.hdr, 34)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t base = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * BN + 128 * h;
            float part[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tmem_ld32(base + 32 * j, r);
                tmem_wait_ld(r);
                // leaves RN(dY * RN(r * r)), two columns a packed multiply (the
                // same bits as scalar ones; 221.1 -> 214.9 us a call)
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float c0 = __uint_as_float(r[i]), c1 = __uint_as_float(r[i + 1]);
                    const float2 rl = make_float2(c0 > 0.0f ? c0 : 0.0f, c1 > 0.0f ? c1 : 0.0f);
                    const uint32_t w = reinterpret_cast<const uint32_t *>(&dy[4 * j + i / 8])[(i % 8) / 2];
                    const float2 pr = mul2(make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)),
                                           mul2(rl, rl));
                    v[i] = pr.x;
                    v[i + 1] = pr.y;
                }
                // levels 1-5 of the N-tile's tree over these 32 columns
#pragma unroll
                for (int s = 1; s < 32; s *= 2)
#pragma unroll
                    for (int i = 0; i + s < 32; i += 2 * s) v[i] = __fadd_rn(v[i], v[i + s]);
                part[j] = v[0];
            }
            // the accumulator is read: the MMA may refill it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
            // levels 6-7, then the partial of (row, N-tile 2 nb + h)
            const float tile = __fadd_rn(__fadd_rn(part[0], part[1]), __fadd_rn(part[2], part[3]));
            if (mine) p.slots[row * n_ntiles + 2 * nb + h] = tile;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

__global__ void __launch_bounds__(256) dsrelu_fold(const DsParams p) {
    if (p.hdr->status != 0) return;  // the GEMM gave up (offsets or a bounded wait): dprob untouched
    const int64_t m = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    if (m >= p.T) return;
    const int n = p.N / 128;
    const float *s = p.slots + m * n;
    float F = __ldcg(s);
    for (int j = 1; j < n; ++j) F = __fadd_rn(F, __ldcg(s + j));
    p.dprob[m] = p.accumulate ? __fadd_rn(p.dprob[m], F) : F;
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

// Map over a row-major bf16 [rows, cols] matrix (cols a multiple of 64) viewed
// as {64 columns, rows, cols / 64 blocks}: a box {64, box_rows, blocks} lands as
// `blocks` consecutive {64, box_rows} atoms, 128-byte swizzle, zero fill past
// the last row.
dgr_status make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t box_rows,
                    uint32_t blocks) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    dgr_status st = encode_fn(&enc);
    if (st != DGR_OK) return st;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols * 2), 128};
    const cuuint32_t box[3] = {64, box_rows, blocks};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DGR_OK : DGR_ERR_CUDA;
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" size_t dgr_dsrelu_dprob_workspace_bytes(int64_t T, int64_t N) {
    if (T < 0 || N < 0 || T > INT32_MAX || N > (1 << 20)) return 0;
    return sizeof(WsHeader) + align_up(static_cast<size_t>(T) * static_cast<size_t>((N + 127) / 128) * 4);
}

namespace dgr {
namespace {

dgr_status dsrelu_call(const void *A, const void *B, const int64_t *d_offs, int32_t E, int64_t T, int64_t K, int64_t N,
                       const void *dY, float *dprob, int32_t accumulate, void *ws, size_t ws_bytes, void *stream,
                       int32_t stall_role, int32_t stall_after, uint64_t stall_ns) {
    if (E < 1 || T < 0 || K < 1 || N < 1) return DGR_ERR_INVALID_ARG;
    if (E > kMaxExperts || T > INT32_MAX || (K % BK) != 0 || (N % BN) != 0 || N > (1 << 20) ||
        static_cast<int64_t>(E) * K > INT32_MAX)
        return DGR_ERR_UNSUPPORTED;
    if (!d_offs || (T > 0 && (!A || !B || !dY || !dprob))) return DGR_ERR_INVALID_ARG;  // T = 0: dprob is empty
    if (!aligned(d_offs, 8) || !aligned(dprob, 4) || (A && !aligned(A, 16)) || (B && !aligned(B, 16)) ||
        (dY && !aligned(dY, 16)))
        return DGR_ERR_MISALIGNED;
    const size_t need = dgr_dsrelu_dprob_workspace_bytes(T, N);
    if (ranges_overlap(dprob, T * 4, A, T * K * 2) || ranges_overlap(dprob, T * 4, B, E * K * N * 2) ||
        ranges_overlap(dprob, T * 4, dY, T * N * 2) || ranges_overlap(dprob, T * 4, d_offs, (E + 1) * 8))
        return DGR_ERR_ALIAS;
    if (T > 0) {
        if (!ws) return DGR_ERR_INVALID_ARG;
        if (ws_bytes < need) return DGR_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(ws, kAlign)) return DGR_ERR_MISALIGNED;
        if (ranges_overlap(dprob, T * 4, ws, need)) return DGR_ERR_ALIAS;
    }
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    if (T == 0) return DGR_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CUtensorMap mA, mB;
    if ((st = make_map(&mA, A, T, K, BM, 1)) != DGR_OK) return st;
    if ((st = make_map(&mB, B, static_cast<int64_t>(E) * K, N, 64, BN / 64)) != DGR_OK) return st;
    DsParams p{};
    p.offs = d_offs;
    p.E = E;
    p.T = static_cast<int32_t>(T);
    p.K = static_cast<int32_t>(K);
    p.N = static_cast<int32_t>(N);
    p.nbs = static_cast<int32_t>(N / BN);
    p.dY = static_cast<const uint16_t *>(dY);
    p.dprob = dprob;
    p.accumulate = accumulate ? 1 : 0;
    p.hdr = static_cast<WsHeader *>(ws);
    p.slots = reinterpret_cast<float *>(static_cast<char *>(ws) + sizeof(WsHeader));
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(dsrelu_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes)) !=
            cudaSuccess)
        return DGR_ERR_CUDA;
    const int64_t tiles_max = ((T + BM - 1) / BM + E) * (N / BN);
    p.sched = sched_setting();
    p.stall_role = stall_role;
    p.stall_after = stall_after;
    p.stall_ns = stall_ns;
    const unsigned grid = sched_grid(static_cast<unsigned>(tiles_max < sms ? tiles_max : sms));
    dsrelu_gemm<<<grid, kThreads, kSmemBytes, s>>>(mA, mB, p);
    if (cudaGetLastError() != cudaSuccess) return DGR_ERR_CUDA;
    dsrelu_fold<<<static_cast<unsigned>((T + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? DGR_OK : DGR_ERR_CUDA;
}

}  // namespace
}  // namespace dgr

extern "C" dgr_status dgr_dsrelu_dprob(const void *A, const void *B, const int64_t *d_offs, int32_t E, int64_t T,
                                       int64_t K, int64_t N, const void *dY, float *dprob, int32_t accumulate,
                                       void *ws, size_t ws_bytes, void *stream) {
    return dsrelu_call(A, B, d_offs, E, T, K, N, dY, dprob, accumulate, ws, ws_bytes, stream, 0, 0, 0);
}

extern "C" dgr_status dgr_diag_dsrelu_stall(const void *A, const void *B, const int64_t *d_offs, int32_t E,
                                            int64_t T, int64_t K, int64_t N, const void *dY, float *dprob,
                                            void *ws, size_t ws_bytes, int32_t role, int32_t after,
                                            int32_t limit_us, void *stream) {
    if (role < 1 || role > 3 || after < 0 || limit_us < 1 || limit_us > 1000000) return DGR_ERR_INVALID_ARG;
    return dsrelu_call(A, B, d_offs, E, T, K, N, dY, dprob, 0, ws, ws_bytes, stream, role, after,
                       static_cast<uint64_t>(limit_us) * 1000ull);
}
