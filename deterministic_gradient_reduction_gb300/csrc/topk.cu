// Canonical compact top-K: per row, the K slots sorted stably by id (padding,
// id < 0, last), the logits permuted alike, and the softmax of the valid
// slots recomputed in that order.
//
// Megatron-LM PR #7441, Source 1: the compact top-K returns the selected ids
// in a run-dependent slot order and accumulates its softmax in that order;
// the fix (_canonicalize_compact_topk) sorts the ids per row with padding
// last, permutes the logits with the same permutation and recomputes the
// softmax in that order; rows that are all padding become 0 rather than NaN.
//
// One warp per row. Lane l owns slots [l*KPL, l*KPL + KPL) (KPL = 1, 2, 4 or
// 8: up to 256 slots). Each slot gets a key that orders (padding, id, slot):
// (id << 8 | slot) in 32 bits when every id of the row is below 2^23 (padding
// as 0xffffff00 | slot), else (id, slot) in 64 bits (padding id 0xffffffff).
// The keys are distinct, so an ascending bitonic sort over 32*KPL positions
// (registers within a lane, xor-shuffles across lanes) gives exactly the
// stable order.
// The row's ids and logits are staged in the warp's shared memory and gathered
// back by slot number. The softmax: m = max valid logit, d = RN(l - m),
// e = exp_tang(d), Z = the canonical sum of e over the sorted valid positions
// (tiles of 128 positions, pairwise inside, ascending fold), p = RN(e / Z).
#include "dgr_common.cuh"

namespace dgr {
namespace {

// The exponential: P. T. P. Tang's table-driven method ("Table-driven
// implementation of the exponential function in IEEE floating-point
// arithmetic", ACM TOMS 15(2), 1989) in binary32, every operation rounded to
// nearest, in a fixed order, so the softmax's bits are those of its
// definition with this exponential:
//   N = nearest integer to x * 32/ln2, j = N mod 32, m = floor(N / 32);
//   r = (x - N L1) + (-(N L2)), L1 = 1419 * 2^-16 (N L1 exact), L2 = ln2/32 - L1;
//   p = r + r^2 (1/2 + r/6);
//   exp(x) = 2^m (S_lead[j] + (S_trail[j] + S p)), S = S_lead[j] + S_trail[j],
//   where S_lead[j] + S_trail[j] = 2^(j/32), S_lead to 18 significant bits.
// The scaling by 2^m is two multiplications by exact powers of two, so a
// subnormal result is rounded once. x < -104 gives +0.0. At most 0.77 ulp
// from exp over every binary32 x in [-104, 0].
__device__ const uint32_t kTangLead[32] = {
    0x3f800000, 0x3f82cd80, 0x3f85aac0, 0x3f889800, 0x3f8b95c0, 0x3f8ea440, 0x3f91c3c0, 0x3f94f500,
    0x3f983800, 0x3f9b8d40, 0x3f9ef540, 0x3fa27040, 0x3fa5fec0, 0x3fa9a140, 0x3fad5840, 0x3fb12400,
    0x3fb50500, 0x3fb8fbc0, 0x3fbd08c0, 0x3fc12c40, 0x3fc56740, 0x3fc9b9c0, 0x3fce2480, 0x3fd2a800,
    0x3fd74500, 0x3fdbfbc0, 0x3fe0ccc0, 0x3fe5b900, 0x3feac0c0, 0x3fefe4c0, 0x3ff52580, 0x3ffa83c0};
__device__ const uint32_t kTangTrail[32] = {
    0x00000000, 0x35531585, 0x34d9f312, 0x35e8092e, 0x3471f546, 0xb54e9746, 0x361b9d59, 0xb602b808,
    0xb5fae724, 0xb548c556, 0xb5d9f6e6, 0x34c0c312, 0x36354d8b, 0x3655a754, 0xb40adeaf, 0xb5a7e2d5,
    0xb5ccc062, 0xb605c4e8, 0xb6630540, 0x35cca667, 0xb62f7558, 0xb49e6474, 0x35c151f8, 0x366c8f89,
    0xb4cd4a59, 0xb5868251, 0x36776155, 0x355cef90, 0x355cfba5, 0xb54c8465, 0xb4bab6de, 0xb5d248dd};

__device__ __forceinline__ float pow2f(int k) {  // -126 <= k <= 127
    return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

__device__ __forceinline__ float exp_tang(float x) {
    const float inv_l = __uint_as_float(0x4238aa3bu);  // 32/ln2
    const float l1 = __uint_as_float(0x3cb16000u);     // 1419 * 2^-16
    const float l2 = __uint_as_float(0x3710bfbfu);     // ln2/32 - l1
    const float a2 = __uint_as_float(0x3e2aaaabu);     // 1/6
    if (x != x) return x;
    if (x < -104.0f) return 0.0f;
    const int n = __float2int_rn(__fmul_rn(x, inv_l));
    const float nf = __int2float_rn(n);
    const float r = __fadd_rn(__fsub_rn(x, __fmul_rn(nf, l1)), -__fmul_rn(nf, l2));
    const float p = __fadd_rn(r, __fmul_rn(__fmul_rn(r, r), __fadd_rn(0.5f, __fmul_rn(r, a2))));
    const int j = n & 31;
    const int m = n >> 5;
    const float sl = __uint_as_float(__ldg(&kTangLead[j]));
    const float st = __uint_as_float(__ldg(&kTangTrail[j]));
    const float S = __fadd_rn(sl, st);
    const float y = __fadd_rn(sl, __fadd_rn(st, __fmul_rn(S, p)));
    const int m1 = m < -100 ? -100 : m;
    return __fmul_rn(__fmul_rn(y, pow2f(m1)), pow2f(m - m1));
}

constexpr int kWarps = 8;
constexpr int kMaxK = 256;

struct TopkParams {
    const int32_t *ids;
    const float *logits;
    int64_t ld_ids, ld_logits, ld_out;
    int64_t R;
    int32_t K;
    int32_t vec;  // K == 32 * KPL and every row 16-byte aligned: a lane's slots move as 16-byte words
    int32_t *out_ids;
    float *out_logits;
    float *probs;
};

__device__ __forceinline__ uint64_t shfl_xor_key(uint64_t v, int m) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint32_t shfl_xor_key(uint32_t v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }

// Ascending bitonic sort of the warp's 32 * KPL keys, position lane * KPL + i.
// A stage (k, j) compares positions p and p ^ j and keeps the smaller at the
// lower position when p & k is 0. With KPL a power of two, a stage with
// j >= KPL pairs lanes lane ^ (j / KPL) and its direction is a property of
// the lane alone; a stage with j < KPL pairs registers of one lane and its
// direction is a bit of i (k < KPL, a constant) or of the lane.
template <int KPL, typename Key>
__device__ __forceinline__ void bitonic(Key (&key)[KPL], int lane) {
    constexpr int N = 32 * KPL;
#pragma unroll
    for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j < KPL) {
                // lanes hold whole k-blocks when k >= KPL: one direction a lane
                const bool lane_desc = k >= KPL && (lane & (k / KPL)) != 0;
#pragma unroll
                for (int i = 0; i < KPL; ++i) {
                    const int q = i ^ j;
                    if (q > i) {
                        const bool desc = k < KPL ? (i & k) != 0 : lane_desc;
                        const Key lo = min(key[i], key[q]), hi = max(key[i], key[q]);
                        key[i] = desc ? hi : lo;
                        key[q] = desc ? lo : hi;
                    }
                }
            } else {
                const int m = j / KPL;  // lane distance
                // keep the smaller when (lower half) == (ascending block)
                const bool take_lo = ((lane & m) == 0) == ((lane & (k / KPL)) == 0);
#pragma unroll
                for (int i = 0; i < KPL; ++i) {
                    const Key o = shfl_xor_key(key[i], m);
                    key[i] = take_lo ? min(key[i], o) : max(key[i], o);
                }
            }
        }
    }
}

template <int KPL>
__global__ void __launch_bounds__(kWarps * 32) topk_kernel(const TopkParams p) {
    __shared__ int32_t s_id[kWarps][kMaxK];
    __shared__ float s_lg[kWarps][kMaxK];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + w;
    if (r >= p.R) return;  // whole warps only: every shuffle below is warp-uniform
    const int K = p.K;
    const int32_t *idr = p.ids + r * p.ld_ids;
    const float *lgr = p.logits + r * p.ld_logits;

    // the row's ids and logits into the warp's shared memory; may the
    // 32-bit keys order this row (every id below 2^23)?
    bool narrow = true;
    if (KPL >= 4 && p.vec) {
#pragma unroll
        for (int i = 0; i < KPL; i += 4) {
            const int s = lane * KPL + i;
            const int4 v = __ldg(reinterpret_cast<const int4 *>(idr + s));
            const float4 f = __ldg(reinterpret_cast<const float4 *>(lgr + s));
            *reinterpret_cast<int4 *>(&s_id[w][s]) = v;
            *reinterpret_cast<float4 *>(&s_lg[w][s]) = f;
            narrow = narrow && v.x < (1 << 23) && v.y < (1 << 23) && v.z < (1 << 23) && v.w < (1 << 23);
        }
    } else {
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const int s = lane * KPL + i;
            if (s < K) {
                const int32_t id = idr[s];
                s_id[w][s] = id;
                s_lg[w][s] = lgr[s];
                narrow = narrow && id < (1 << 23);
            }
        }
    }
    narrow = __all_sync(0xffffffffu, narrow);
    __syncwarp();
    // sorted slot numbers and validity, position lane * KPL + i
    int slot[KPL];
    bool valid[KPL];
    if (narrow) {
        uint32_t key[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const int s = lane * KPL + i;
            key[i] = ~0u;  // positions past K sort after everything
            if (s < K) {
                const int32_t id = s_id[w][s];
                key[i] = ((id < 0 ? 0xffffffu : static_cast<uint32_t>(id)) << 8) | static_cast<uint32_t>(s);
            }
        }
        bitonic<KPL>(key, lane);
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            slot[i] = static_cast<int>(key[i] & 0xffu);
            valid[i] = (key[i] >> 8) != 0xffffffu;
        }
    } else {
        uint64_t key[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const int s = lane * KPL + i;
            key[i] = ~0ull;
            if (s < K) {
                const int32_t id = s_id[w][s];
                const uint32_t hi = id < 0 ? 0xffffffffu : static_cast<uint32_t>(id);
                key[i] = (static_cast<uint64_t>(hi) << 32) | static_cast<uint32_t>(s);
            }
        }
        bitonic<KPL>(key, lane);
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            slot[i] = static_cast<int>(key[i] & 0xffffffffu);
            valid[i] = (key[i] >> 32) != 0xffffffffull;
        }
    }

    // gather the sorted slots; n = valid slots (they come first)
    int32_t oid[KPL];
    float olg[KPL];
    int my_valid = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const int pos = lane * KPL + i;
        oid[i] = 0;
        olg[i] = 0.0f;
        if (pos < K) {
            oid[i] = s_id[w][slot[i]];
            olg[i] = s_lg[w][slot[i]];
            my_valid += valid[i] ? 1 : 0;
        }
    }
    int n = my_valid;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) n += __shfl_xor_sync(0xffffffffu, n, s);

    // the softmax of the valid positions [0, n), in sorted order
    float e[KPL];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < KPL; ++i)
        if (lane * KPL + i < n) m = fmaxf(m, olg[i]);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
#pragma unroll
    for (int i = 0; i < KPL; ++i) e[i] = lane * KPL + i < n ? exp_tang(__fsub_rn(olg[i], m)) : 0.0f;
    // tile partials: the lane's KPL positions (pairwise, absent past n), then
    // lanes pairwise up to a tile of 128 positions (128 / KPL lanes)
    constexpr int kTileLanes = 128 / KPL < 32 ? 128 / KPL : 32;
    const int n_lane = max(0, min(KPL, n - lane * KPL));
    float acc[KPL][1];
#pragma unroll
    for (int i = 0; i < KPL; ++i) acc[i][0] = e[i];
#pragma unroll
    for (int s = 1; s < KPL; s *= 2) {
#pragma unroll
        for (int i = 0; i + s < KPL; i += 2 * s)
            if (i + s < n_lane) acc[i][0] = __fadd_rn(acc[i][0], acc[i + s][0]);
    }
    float t = acc[0][0];
    bool present = n_lane > 0;
#pragma unroll
    for (int s = 1; s < kTileLanes; s *= 2) {
        const bool left_is_me = (lane & s) == 0;
        const float o = __shfl_xor_sync(0xffffffffu, t, s);
        const bool o_present = __shfl_xor_sync(0xffffffffu, present ? 1 : 0, s) != 0;
        const bool left_present = left_is_me ? present : o_present;
        const bool right_present = left_is_me ? o_present : present;
        if (left_present && right_present) t = __fadd_rn(t, o);
        else if (!left_is_me && left_present) t = o;
        present = left_present;
    }
    // ascending fold of the tiles (first lane of each tile holds its partial)
    constexpr int kTiles = 32 / kTileLanes;
    float Z = __shfl_sync(0xffffffffu, t, 0);
#pragma unroll
    for (int q = 1; q < kTiles; ++q) {
        const float tq = __shfl_sync(0xffffffffu, t, q * kTileLanes);
        if (q * 128 < n) Z = __fadd_rn(Z, tq);
    }

    int32_t *oi = p.out_ids + r * p.ld_out;
    float *ol = p.out_logits + r * p.ld_out;
    float *op = p.probs + r * p.ld_out;
    float pr[KPL];
#pragma unroll
    for (int i = 0; i < KPL; ++i) pr[i] = lane * KPL + i < n ? __fdiv_rn(e[i], Z) : 0.0f;
    if (KPL >= 4 && p.vec) {
#pragma unroll
        for (int i = 0; i < KPL; i += 4) {
            const int pos = lane * KPL + i;
            *reinterpret_cast<int4 *>(oi + pos) = make_int4(oid[i], oid[i + 1], oid[i + 2], oid[i + 3]);
            *reinterpret_cast<float4 *>(ol + pos) = make_float4(olg[i], olg[i + 1], olg[i + 2], olg[i + 3]);
            *reinterpret_cast<float4 *>(op + pos) = make_float4(pr[i], pr[i + 1], pr[i + 2], pr[i + 3]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const int pos = lane * KPL + i;
            if (pos < K) {
                oi[pos] = oid[i];
                ol[pos] = olg[i];
                op[pos] = pr[i];
            }
        }
    }
}

template <int KPL>
dgr_status launch_topk(const TopkParams &p, cudaStream_t s) {
    const int64_t grid = (p.R + kWarps - 1) / kWarps;
    topk_kernel<KPL><<<static_cast<unsigned>(grid), kWarps * 32, 0, s>>>(p);
    return launch_status();
}

}  // namespace
}  // namespace dgr

using namespace dgr;

extern "C" dgr_status dgr_topk_canonicalize(const int32_t *ids, int64_t ld_ids, const float *logits,
                                            int64_t ld_logits, int64_t R, int32_t K, int32_t *out_ids,
                                            float *out_logits, float *probs, int64_t ld_out, void *stream) {
    if (R < 0 || K < 1 || ld_ids < K || ld_logits < K || ld_out < K) return DGR_ERR_INVALID_ARG;
    if (K > kMaxK || R > (static_cast<int64_t>(INT32_MAX) - 1) * kWarps) return DGR_ERR_UNSUPPORTED;
    if (R > 0 && (!ids || !logits || !out_ids || !out_logits || !probs)) return DGR_ERR_INVALID_ARG;
    if (!aligned(ids, 4) || !aligned(logits, 4) || !aligned(out_ids, 4) || !aligned(out_logits, 4) ||
        !aligned(probs, 4))
        return DGR_ERR_MISALIGNED;
    if (R > 0) {
        const size_t in_i = static_cast<size_t>(((R - 1) * ld_ids + K) * 4);
        const size_t in_l = static_cast<size_t>(((R - 1) * ld_logits + K) * 4);
        const size_t out = static_cast<size_t>(((R - 1) * ld_out + K) * 4);
        const void *outs[3] = {out_ids, out_logits, probs};
        for (int a = 0; a < 3; ++a) {
            if (ranges_overlap(outs[a], out, ids, in_i) || ranges_overlap(outs[a], out, logits, in_l))
                return DGR_ERR_ALIAS;
            for (int b = a + 1; b < 3; ++b)
                if (ranges_overlap(outs[a], out, outs[b], out)) return DGR_ERR_ALIAS;
        }
    }
    dgr_status st = check_device();
    if (st != DGR_OK) return st;
    if (R == 0) return DGR_OK;
    TopkParams p{};
    p.ids = ids;
    p.logits = logits;
    p.ld_ids = ld_ids;
    p.ld_logits = ld_logits;
    p.ld_out = ld_out;
    p.R = R;
    p.K = K;
    p.out_ids = out_ids;
    p.out_logits = out_logits;
    p.probs = probs;
    const int kpl = K <= 32 ? 1 : K <= 64 ? 2 : K <= 128 ? 4 : 8;
    p.vec = (K == 32 * kpl && kpl >= 4 && aligned(ids, 16) && aligned(logits, 16) && aligned(out_ids, 16) &&
             aligned(out_logits, 16) && aligned(probs, 16) && ld_ids % 4 == 0 && ld_logits % 4 == 0 &&
             ld_out % 4 == 0)
                ? 1
                : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K <= 32) return launch_topk<1>(p, s);
    if (K <= 64) return launch_topk<2>(p, s);
    if (K <= 128) return launch_topk<4>(p, s);
    return launch_topk<8>(p, s);
}
