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

#ifdef __cplusplus
}
#endif

#endif /* DGR_DIAG_H */
