// Deterministic aux-loss scalar: aux = RN(scale * S),
//   x[t] = fold over expert tiles of pw_128( RN(probs[t][e] * tpe[e]) ),
//   S    = fold over token tiles of pw_128( x[t] ).
//
// Megatron-LM PR #7441, Source 5: the fused router aux loss reduces its scalar
// with a cross-block float atomicAdd; its gradient is the closed form
// coeff*E/(topk*N^2)*tokens_per_expert[e], so the loss is that factor (the
// caller's `scale`) times the sum over tokens and experts of
// probs * tokens_per_expert, taken here in the canonical order: each token's
// row dot (expert tiles of 128), then the column sum of one column over the
// tokens (token tiles of 128).
//
// One launch: one 8-warp CTA per tile of 128 tokens. Warp w owns tokens
// [16w, 16w + 16): their rows' loads all in flight, then per token a lane's 4
// products summed in registers and the expert tile's upper levels by
// xor-shuffles, expert tiles folded in order; the 16 token values by
// shuffles, the 8 warps' by thread 0: the tile's partial to its slot. The CTA
// then fences its slot and takes an integer ticket; the CTA with the last
// ticket stages all slots in shared memory and folds them in ascending tile
// order on one thread, times scale, into the output scalar, and resets the
// ticket for the next call.
#include "dgr_common.cuh"

namespace dgr {
namespace {

constexpr int kTileThreads = 256;
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kTokPerWarp = 128 / kTileWarps;  // 16
constexpr int kMaxExperts = 1024;
constexpr int kFoldChunk = 2048;  // slots staged at a time by the last CTA

struct AuxParams {
    const float *probs;
    int64_t N, ld;
    int32_t E;
    int32_t vec;  // rows 16-byte aligned, E a multiple of 4: a lane's 4 experts as one 16-byte load
    const int32_t *tpe;
    float scale;
    float *out;
    float *slots;  // [ceil(N / 128)]
    WsHeader *hdr;  // pad[0]: tiles done (ticket)
    int32_t n_tiles;
    Sched sched;    // which CTA takes which token tile
};

// Pairwise levels across lanes: lanes [0, 32) hold aligned leaf groups whose
// presence is a prefix (lane l present iff l < n_present); distances 1 .. L/2.
// Lane 0 ends with the root of lanes [0, L).
template <int L>
__device__ __forceinline__ float lane_tree(float v, int lane, int n_present) {
    bool present = lane < n_present;
#pragma unroll
    for (int s = 1; s < L; s *= 2) {
        const bool left_is_me = (lane & s) == 0;
        const float o = __shfl_xor_sync(0xffffffffu, v, s);
        const bool o_present = __shfl_xor_sync(0xffffffffu, present ? 1 : 0, s) != 0;
        const bool left_present = left_is_me ? present : o_present;
        const bool right_present = left_is_me ? o_present : present;
        if (left_present && right_present) v = __fadd_rn(v, o);
        else if (!left_is_me && left_present) v = o;
        present = left_present;
    }
    return v;
}

__global__ void __launch_bounds__(kTileThreads, 3) aux_tiles(const AuxParams p) {
    __shared__ float wpart[kTileWarps];
    __shared__ float tpe_f[kMaxExperts];
    __shared__ float stage[kFoldChunk];
    __shared__ int last;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    if (p.N == 0) {  // an empty sum
        if (tid == 0) *p.out = __fmul_rn(p.scale, 0.0f);
        return;
    }
    for (int e = tid; e < p.E; e += kTileThreads) tpe_f[e] = static_cast<float>(p.tpe[e]);
    __syncthreads();
    // token tiles in the schedule's order; with a capped grid a CTA takes several
    for (int32_t it = blockIdx.x; it < p.n_tiles; it += gridDim.x) {
        const int32_t tile = static_cast<int32_t>(sched_item(p.sched, static_cast<uint32_t>(it)));
        const int64_t t0 = static_cast<int64_t>(tile) * 128;
        const int count = static_cast<int>(min(static_cast<int64_t>(128), p.N - t0));  // tokens in this tile
        const int n_mine = max(0, min(kTokPerWarp, count - w * kTokPerWarp));
        const int e_tiles = (p.E + 127) / 128;
        float xs = 0.0f;  // lane i < 16: token 16w + i's row dot
        for (int k = 0; k < e_tiles; ++k) {
            const int e0 = k * 128 + lane * 4;
            const int n_e = max(0, min(4, p.E - e0));               // this lane's experts
            const int lanes_present = (min(128, p.E - k * 128) + 3) / 4;  // lanes with an expert
            float tw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) tw[i] = i < n_e ? tpe_f[e0 + i] : 0.0f;
            // the rows' loads all in flight (predicated inside the load, so
            // nothing waits for one before issuing the next)
            float4 row[kTokPerWarp];
            const bool whole = p.vec && n_e == 4;
#pragma unroll
            for (int r = 0; r < kTokPerWarp; ++r) {
                row[r] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                const float *src = p.probs + (t0 + w * kTokPerWarp + r) * p.ld + e0;
                ldg_nc_v4f_if(row[r], src, whole && r < n_mine);
                if (!whole && r < n_mine) {
                    if (n_e > 0) row[r].x = __ldg(src);
                    if (n_e > 1) row[r].y = __ldg(src + 1);
                    if (n_e > 2) row[r].z = __ldg(src + 2);
                    if (n_e > 3) row[r].w = __ldg(src + 3);
                }
            }
            // every token's 4 leaves: (0 + 1) + (2 + 3), absent past E
            float v[kTokPerWarp];
#pragma unroll
            for (int r = 0; r < kTokPerWarp; ++r) {
                const float a = __fmul_rn(row[r].x, tw[0]), b = __fmul_rn(row[r].y, tw[1]);
                const float c = __fmul_rn(row[r].z, tw[2]), d = __fmul_rn(row[r].w, tw[3]);
                v[r] = a;
                if (n_e > 1) v[r] = __fadd_rn(a, b);
                if (n_e > 3) v[r] = __fadd_rn(v[r], __fadd_rn(c, d));
                else if (n_e > 2) v[r] = __fadd_rn(v[r], c);
            }
            // the expert tile's upper levels, all 16 tokens at once (the lanes'
            // presence is the experts', the same for every token)
            bool present = lane < lanes_present;
#pragma unroll
            for (int s = 1; s < 32; s *= 2) {
                const bool left_is_me = (lane & s) == 0;
                const bool o_present = __shfl_xor_sync(0xffffffffu, present ? 1 : 0, s) != 0;
                const bool left_present = left_is_me ? present : o_present;
                const bool right_present = left_is_me ? o_present : present;
#pragma unroll
                for (int r = 0; r < kTokPerWarp; ++r) {
                    const float o = __shfl_xor_sync(0xffffffffu, v[r], s);
                    if (left_present && right_present) v[r] = __fadd_rn(v[r], o);
                    else if (!left_is_me && left_present) v[r] = o;
                }
                present = left_present;
            }
            // lane 0 holds every token's tile value: token r's goes to lane r
            float mine = 0.0f;
#pragma unroll
            for (int r = 0; r < kTokPerWarp; ++r) {
                const float tr = __shfl_sync(0xffffffffu, v[r], 0);
                if (lane == r) mine = tr;
            }
            if (lane < n_mine) xs = k == 0 ? mine : __fadd_rn(xs, mine);
        }
        // the warp's 16 token values (an aligned subtree of the token tile)
        const float wv = lane_tree<kTokPerWarp>(lane < kTokPerWarp ? xs : 0.0f, lane, n_mine);
        if (lane == 0) wpart[w] = wv;
        __syncthreads();
        if (tid == 0) {
            // warps pairwise: (0, 1), (2, 3), ... then (0, 2), ... then (0, 4);
            // warp q present iff it has a token
            const int nw = (count + kTokPerWarp - 1) / kTokPerWarp;
            float u[kTileWarps];
#pragma unroll
            for (int q = 0; q < kTileWarps; ++q) u[q] = wpart[q];
#pragma unroll
            for (int s = 1; s < kTileWarps; s *= 2) {
#pragma unroll
                for (int q = 0; q + s < kTileWarps; q += 2 * s)
                    if (q + s < nw) u[q] = __fadd_rn(u[q], u[q + s]);
            }
            p.slots[tile] = u[0];
            __threadfence();  // the slot before the ticket
            last = atomicAdd(&p.hdr->pad[0], 1) == p.n_tiles - 1;
        }
        __syncthreads();
        if (!last) {
            __syncthreads();  // wpart and last are reused by the CTA's next tile
            continue;
        }
        // every tile fenced its slot before its ticket (the CTA taking the last
        // ticket has no tile left): fold them all
        __threadfence();
        const int64_t n = p.n_tiles;
        float F = 0.0f;
        for (int64_t c0 = 0; c0 < n; c0 += kFoldChunk) {
            const int m = static_cast<int>(min(static_cast<int64_t>(kFoldChunk), n - c0));
            for (int i = tid; i < m; i += kTileThreads) stage[i] = __ldcg(p.slots + c0 + i);
            __syncthreads();
            if (tid == 0)
                for (int i = 0; i < m; ++i) F = (c0 + i == 0) ? stage[i] : __fadd_rn(F, stage[i]);
            __syncthreads();
        }
        if (tid == 0) {
            *p.out = __fmul_rn(p.scale, F);
            p.hdr->pad[0] = 0;  // ready for the next call
        }
        return;
    }
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" size_t dgr_aux_loss_workspace_bytes(int64_t N) {
    if (N < 0 || N > INT32_MAX) return 0;
    return sizeof(WsHeader) + align_up(static_cast<size_t>((N + 127) / 128) * 4);
}

extern "C" dgr_status dgr_aux_loss(const float *probs, int64_t N, int32_t E, int64_t ld,
                                   const int32_t *d_tokens_per_expert, float scale, float *d_out, void *ws,
                                   size_t ws_bytes, void *stream) {
    if (N < 0 || E < 1 || ld < E || !d_out || !d_tokens_per_expert) return DGR_ERR_INVALID_ARG;
    if (E > kMaxExperts || N > INT32_MAX) return DGR_ERR_UNSUPPORTED;
    if (N > 0 && !probs) return DGR_ERR_INVALID_ARG;
    if (!aligned(d_out, 4) || !aligned(d_tokens_per_expert, 4) || (probs && !aligned(probs, 4)))
        return DGR_ERR_MISALIGNED;
    const size_t need = dgr_aux_loss_workspace_bytes(N);
    const size_t probs_bytes = N > 0 ? static_cast<size_t>(((N - 1) * ld + E) * 4) : 0;
    if (ranges_overlap(d_out, 4, probs, probs_bytes) || ranges_overlap(d_out, 4, d_tokens_per_expert, E * 4))
        return DGR_ERR_ALIAS;
    if (N > 0) {
        if (!ws) return DGR_ERR_INVALID_ARG;
        if (ws_bytes < need) return DGR_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(ws, kAlign)) return DGR_ERR_MISALIGNED;
        if (ranges_overlap(d_out, 4, ws, need)) return DGR_ERR_ALIAS;
    }
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    AuxParams p{};
    p.probs = probs;
    p.N = N;
    p.ld = ld;
    p.E = E;
    p.vec = (aligned(probs, 16) && ld % 4 == 0) ? 1 : 0;
    p.tpe = d_tokens_per_expert;
    p.scale = scale;
    p.out = d_out;
    p.slots = ws ? reinterpret_cast<float *>(static_cast<char *>(ws) + sizeof(WsHeader)) : nullptr;
    p.hdr = ws ? static_cast<WsHeader *>(ws) : nullptr;
    const int64_t tiles = N > 0 ? (N + 127) / 128 : 1;  // N = 0: one CTA writes scale * +0.0
    p.n_tiles = static_cast<int32_t>(tiles);
    p.sched = sched_for(static_cast<uint32_t>(tiles));
    aux_tiles<<<sched_grid(static_cast<unsigned>(tiles)), kTileThreads, 0, s>>>(p);
    return launch_status();
}
