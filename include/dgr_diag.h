/*
 * dgr_diag.h - diagnostics of the dgr library (GB300, sm_103a).
 *
 * Not part of the reduction path. These entries exist so that tests can
 * check the assumptions the path rests on against the hardware itself.
 */
#ifndef DGR_DIAG_H
#define DGR_DIAG_H

#include <stddef.h>
#include <stdint.h>

#include "dgr.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One tensor-core K16 step (tcgen05.mma kind::f16, bf16 inputs, fp32
 * accumulator, M = 128, N = 256) per problem: D = C + A B (accumulate != 0)
 * or D = A B (accumulate = 0, the accumulator input disabled, as on the first
 * step of a wgrad chunk). The operands are placed in shared memory with the
 * same MN-major 128-byte-swizzle layout and descriptors as the grouped wgrad
 * kernel's pipeline stages.
 *
 * The grouped wgrad of FlashInfer PR #8924 ("Design and numerics") fixes the
 * split order but not the arithmetic inside one tensor-core step; the tests
 * use this entry to check the oracle's model of that step bit for bit, in
 * the manner of Fasi, Higham, Mikaitis and Pranesh, "Numerical behavior of
 * NVIDIA tensor cores" (PeerJ CS 7:e330, 2021).
 *
 * A: [n_prob][128][16] bf16 bits (row m, column k), B: [n_prob][16][256] bf16
 * bits (row k, column n), C, D: [n_prob][128][256] fp32; device pointers.
 * ws: at least 256 bytes, zeroed (status word, see dgr_read_device_status()).
 */
dgr_status dgr_tc_probe_k16(const uint16_t *A, const uint16_t *B, const float *C, float *D, int32_t n_prob,
                            int32_t accumulate, void *ws, size_t ws_bytes, void *stream);

/*
 * A bounded wait that runs out, on purpose: one kernel waits, through the
 * library's own wait helper, for something that nothing will ever complete,
 * and gives up after limit_us microseconds instead of the path's 2 s. which =
 * 0: the integer-counter wait of the column-sum folders and index_add fold
 * blocks (on a workspace word nobody increments); which = 1: the mbarrier wait
 * of the tensor-core pipelines (on a fresh barrier nobody arrives at). The
 * kernel records DGR_ERR_TIMEOUT in the workspace status word (where = 90 + which)
 * and returns; the context stays usable. No GPU fault or hang is involved.
 * ws: at least 256 bytes, zeroed. limit_us: 1 .. 1,000,000.
 */
dgr_status dgr_diag_wait_timeout(int32_t which, int32_t limit_us, void *ws, size_t ws_bytes, void *stream);

/*
 * The same timeout on the status word of the no-alloc column sum's static
 * array (its 256-byte header is zeroed first, on `stream`): afterwards
 * dgr_colsum_noalloc_read_status() returns DGR_ERR_TIMEOUT, as it would after
 * a column-sum folder gave up. Shares the array with every no-alloc call.
 */
dgr_status dgr_diag_noalloc_wait_timeout(int32_t which, int32_t limit_us, void *stream);

/*
 * The grouped wgrad (dgr_grouped_wgrad_accumulate, same arguments and checks,
 * chunk_tokens 512) with one of CTA 0's roles made to time out inside the
 * tensor-core pipeline: role 1, the TMA producer, before its after-th stage
 * copy; role 2, the MMA issuer, before its after-th stage; role 3, epilogue
 * warp 4, at its after-th tile end (before that tile's reduce-adds). The role
 * waits, bounded by limit_us, on an mbarrier nobody arrives at, records
 * DGR_ERR_TIMEOUT (where = 14 + role) and sets the CTA's abort flag; the CTA's
 * other roles give up their waits, the producer waits (bounded) for its copies
 * in flight, the MMA issuer for the completion of the MMAs it issued, the
 * epilogue for its reduce-adds, and only then is TMEM freed and the CTA done.
 * The other CTAs finish their tiles. main_grad is left partly updated (the
 * stalled CTA's tiles); no GPU fault or hang is involved, and the context
 * stays usable. role: 1 .. 3; after >= 0 (a count never reached: no stall);
 * limit_us: 1 .. 1,000,000.
 */
dgr_status dgr_diag_wgrad_stall(const void *G, const void *X, const int64_t *d_offs, int32_t E, int64_t T_total,
                                int64_t N, int64_t K, float *main_grad, void *ws, size_t ws_bytes, int32_t role,
                                int32_t after, int32_t limit_us, void *stream);

/*
 * The same for the dsReLU dprob GEMM (dgr_dsrelu_dprob, same arguments and
 * checks, accumulate 0): role 1, CTA 0's TMA producer, before its after-th
 * stage copy; role 2, its MMA issuer, before its after-th stage; role 3,
 * epilogue warp 4, before its after-th accumulator. DGR_ERR_TIMEOUT is
 * recorded with where = 40 + role; the CTA drains as the wgrad's does, the
 * other CTAs and the fold launch run to the end, dprob is left invalid, and
 * the context stays usable.
 */
dgr_status dgr_diag_dsrelu_stall(const void *A, const void *B, const int64_t *d_offs, int32_t E, int64_t T, int64_t K,
                                 int64_t N, const void *dY, float *dprob, void *ws, size_t ws_bytes, int32_t role,
                                 int32_t after, int32_t limit_us, void *stream);

/*
 * The packed binary32 arithmetic the kernels use (add.rn.f32x2,
 * mul.rn.f32x2), exposed so that a test can pin it: for i < n_pairs,
 * sum[2i..2i+1] = a + b and prod[2i..2i+1] = a * b, each half rounded to
 * nearest even with subnormals kept, which is what the kernels' bit-exactness
 * rests on. Device pointers of 2 * n_pairs floats, 8-byte aligned.
 */
dgr_status dgr_diag_packed_ops(const float *a, const float *b, int64_t n_pairs, float *sum, float *prod,
                               void *stream);

/*
 * A packed product feeding scalar round-to-nearest adds, the form the dsReLU
 * leaves take: chain[2i..2i+1] = c + RN(a * b), the product by mul.rn.f32x2,
 * each add a separate binary32 add. (A packed product feeding a packed add is
 * not used anywhere: the code generator fuses that pair into a fused
 * multiply-add, which changes the bits.)
 */
dgr_status dgr_diag_packed_chain(const float *a, const float *b, const float *c, int64_t n_pairs, float *chain,
                                 void *stream);

/*
 * How dgr_ordered_colsum() would launch a call of T tokens and H columns,
 * computed on the host alone (no device needed): plan[0] = path (0: at most
 * 512 tiles of 16-byte-vector shapes, one launch whose last warp folds; 1:
 * warp producers and folder CTAs; 2: CTA producers and folder CTAs; -1: T = 0,
 * nothing launched),
 * plan[1] = launches (1, or 2 when the folders, which wait for the producers,
 * could not all be resident beside at least one producer: producers first,
 * folders second), plan[2] = producer CTAs, plan[3] = folder CTAs. vec_ok:
 * whether 16-byte loads apply (x, strides and H aligned to 16 bytes). sms:
 * SMs usable at once; cta_occupancy: CTAs of the path-2 kernel an SM holds;
 * grid_cap: as for dgr_diag_set_schedule (0 = none).
 */
dgr_status dgr_diag_colsum_plan(int64_t T, int64_t H, int32_t tile_rows, int32_t dtype, int32_t vec_ok, int32_t sms,
                                int32_t cta_occupancy, int32_t grid_cap, int32_t *plan);

/*
 * Test-only: how every later launch of this process hands out its work. The
 * kernels take work items (tiles, rows, token chunks, warp shares) in
 * ascending order over as many CTAs as they need; here a test can ask for
 * order = 1 (descending) or 2 (shuffled: item i -> (a i + b) mod n with a
 * coprime to n, a and b derived from seed), and for grid_cap > 0: no launch
 * takes more than grid_cap CTAs (persistent kernels then have fewer CTAs and
 * one-CTA-per-item kernels loop over their items; the column sum switches to
 * its two-launch form when its folders and producers could not all be
 * resident). Bits of every output must not change. (0, 0, 0) restores the
 * default. Process-wide; not for use while other threads launch.
 */
dgr_status dgr_diag_set_schedule(int32_t order, uint32_t seed, int32_t grid_cap);

/*
 * Non-deterministic controls, for tests only: the reductions the pages
 * replace, whose parts meet in float atomicAdds (Megatron-LM PR #8244: the
 * default path's atomics across programs; cuDNN-frontend PR #521: dprob's
 * inter-CTA atomics). A replay test that passes says something only if these
 * change bits from run to run on the same data.
 *   dgr_diag_atomic_colsum: out[h] = sum over t of x[t][h], x bf16 [T, H]
 *     row-major (H <= 4096); one CTA per 128 rows, each adds its column
 *     partials to out (zeroed first, on `stream`) with atomicAdd.
 *   dgr_diag_atomic_rowdot: dprob[m] = sum over n of dY[m][n] Y[m][n], bf16
 *     [M, N] row-major (M <= 524280); one CTA per (128-column tile, 8 rows),
 *     the tile the fastest grid index, each tile's partial added to dprob[m]
 *     (zeroed first) with atomicAdd.
 */
dgr_status dgr_diag_atomic_colsum(const uint16_t *x, int64_t T, int32_t H, float *out, void *stream);
dgr_status dgr_diag_atomic_rowdot(const uint16_t *dY, const uint16_t *Y, int64_t M, int32_t N, float *dprob,
                                  void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DGR_DIAG_H */
