/*
 * dgr.h - deterministic, atomic-free gradient reduction on GB300 (sm_103a).
 *
 * A small C ABI over hand-written CUDA kernels. Every reduction writes FP32
 * partial sums with exactly one writer per partial, then reduces them in one
 * canonical order: a fixed-width pairwise tree inside each tile (adjacent
 * halves; leaves past a ragged end are absent), the tile partials folded in
 * ascending tile order, and the result either written or added to the output
 * with one IEEE binary32 rounding. Results are therefore bitwise identical
 * from run to run, whatever the launch order, grid size or concurrent streams.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns
 *     every buffer (inputs, outputs, workspace). The library allocates no
 *     memory and keeps no state between calls (the one exception,
 *     dgr_ordered_colsum_noalloc, uses a static device scratch; see there).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). All work is enqueued on it; no operation synchronises the host
 *     (the status reads, dgr_read_device_status and dgr_query_device_status,
 *     synchronise their stream to return the word).
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns an error code and launches nothing.
 *   - Workspaces: query the size with the matching *_workspace_bytes() call,
 *     allocate at least that many bytes (256-byte aligned) and ZERO them once
 *     before first use. Every successful call leaves its workspace ready for
 *     the next call with the same sizes (all counters back to zero); its
 *     layout depends on the sizes, so before a call with other sizes it must
 *     be zeroed again (unless the operation's entry allows that change).
 *     One workspace must not be used by two calls that can run at the same
 *     time on the GPU.
 *   - Device-side anomalies (a bounded wait that ran out) are recorded in the
 *     workspace's status word, read with dgr_read_device_status(). After such
 *     an error the outputs of that call are unspecified and the workspace must
 *     be zeroed again before reuse.
 *   - Floating point: binary32 round-to-nearest-even, subnormals kept, no
 *     fused multiply-add anywhere in a reduction.
 *   - Only devices of compute capability 10.3 (sm_103a, GB300) are supported;
 *     on others every launching entry returns DGR_ERR_UNSUPPORTED.
 */
#ifndef DGR_H
#define DGR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t dgr_status;

#define DGR_OK 0
#define DGR_ERR_INVALID_ARG 1          /* a size, stride, flag or pointer is invalid */
#define DGR_ERR_UNSUPPORTED 2          /* device is not sm_103a, or a size is beyond a stated limit */
#define DGR_ERR_WORKSPACE_TOO_SMALL 3  /* ws_bytes below the *_workspace_bytes() figure */
#define DGR_ERR_ALIAS 4                /* an output overlaps an input or the workspace */
#define DGR_ERR_MISALIGNED 5           /* a pointer or stride breaks a stated alignment */
#define DGR_ERR_CUDA 6                 /* a CUDA runtime call failed (launch, attribute) */
#define DGR_ERR_TIMEOUT 7              /* device status: a bounded wait ran out */

#define DGR_DTYPE_F32 0
#define DGR_DTYPE_BF16 1

/* Human-readable name of a status code (static storage). */
const char *dgr_status_string(dgr_status s);

/* Library ABI version (major * 100 + minor). 1.01 added sections 5-8 (grouped
 * dbias, canonical top-K, aux-loss scalar, dsReLU dprob); 1.02 added
 * dgr_query_device_status; 1.03 added dgr_colsum_noalloc_read_status;
 * earlier entries unchanged. */
int32_t dgr_version(void);

/* DGR_OK when `device` is a compute capability 10.3 GPU, else DGR_ERR_UNSUPPORTED. */
dgr_status dgr_device_supported(int32_t device);

/*
 * Copies the status word of a workspace to *status (host pointer) after
 * synchronising `stream`; with clear != 0 it then zeroes the word.
 * DGR_OK in *status means no device-side error was recorded.
 */
dgr_status dgr_read_device_status(const void *ws, int32_t clear, int32_t *status, void *stream);

/*
 * The same read as a return value: synchronises `stream` and returns the
 * status recorded in the workspace's status word (DGR_OK when none was, e.g.
 * DGR_ERR_TIMEOUT after a bounded wait ran out), or the error of the read
 * itself (DGR_ERR_INVALID_ARG for a null ws, DGR_ERR_CUDA). The word is left
 * as it is: clear it with dgr_read_device_status(ws, 1, ...).
 */
dgr_status dgr_query_device_status(const void *ws, void *stream);

/* ------------------------------------------------------------------------ */
/* 1. Ordered column sum                                                     */
/* ------------------------------------------------------------------------ */
/*
 * Megatron-LM PR #8244 ("ordered reduction for the fused pre-GDR gate
 * backward"), description: each program writes independent FP32 partial sums
 * (here one slot row per tile of `tile_rows` tokens) and the caller reduces
 * them in order on the same stream - the A_log / dt_bias-style bias gradient.
 *
 *   out[h] = fold_j pw_W( x[t][h] : t in tile j ),   W = tile_rows,
 *   tokens flattened t = b*S + s, x[b][s][h] at element offset
 *   b*stride_b + s*stride_s + h (the last dimension is contiguous).
 *
 * x:        [B, S, H] elements of `dtype` (DGR_DTYPE_BF16 or DGR_DTYPE_F32).
 * out:      [H] fp32. accumulate = 0 overwrites, else out[h] = out[h] + F.
 *           With B*S = 0 overwrite writes +0.0 and accumulate leaves out.
 * tile_rows: power of two, 1 .. 4096 (128 is the canonical tile).
 * Limits:   H <= 4096; B*S <= 2^31 - 1.
 * Alignment: 16-byte vector loads are used when x, stride_b, stride_s and H
 *           allow it; otherwise a scalar path runs (same bits).
 * ws:       dgr_colsum_workspace_bytes(B*S, H, tile_rows) bytes, zeroed once.
 *           Holds the [tiles, H] FP32 slots and the ready counters.
 * out must not overlap x or ws.
 * Residency: above 512 tiles (of the 16-byte-vector shapes; every tile count
 * for the others) folder CTAs wait, bounded, for producer CTAs of the same
 * launch, so both must be resident together. The call sizes that launch by
 * the SMs usable at once (the device's, or the SM partition of a green
 * context) and, where the folders and one producer would not fit, runs the
 * producers and then the folders as two launches. A share of the GPU the
 * driver does not report (e.g. an MPS active-thread percentage) can still
 * starve the producers: the folders then give up after 2 s and record
 * DGR_ERR_TIMEOUT in the status word; out is then unspecified.
 */
size_t dgr_colsum_workspace_bytes(int64_t T, int64_t H, int32_t tile_rows);
dgr_status dgr_ordered_colsum(const void *x, int32_t dtype, int64_t B, int64_t S, int64_t H,
                              int64_t stride_b, int64_t stride_s, float *out, int32_t accumulate,
                              int32_t tile_rows, void *ws, size_t ws_bytes, void *stream);

/*
 * The same column sum for callers that cannot allocate device memory where
 * they call it (inside another allocator, in a plugin given only input and
 * output pointers, or on a path where a cudaMalloc would stall the device).
 * The pages have no counterpart: this form exists for those callers only.
 *
 * Arguments and results are those of dgr_ordered_colsum() without ws and
 * ws_bytes. The scratch is a static device array of
 * DGR_COLSUM_NOALLOC_SCRATCH_BYTES inside the library (present on every GPU
 * that loads it, until the process exits); nothing is allocated. A call whose
 * dgr_colsum_workspace_bytes(B*S, H, tile_rows) exceeds that size returns
 * DGR_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 * Every argument is checked before the array is touched: a refused call
 * enqueues nothing. The first call on a device looks up the array's device
 * address (with that device current; a lookup that fails is tried again on
 * the next call). Each call then zeroes the part of the array it uses, the whole
 * dgr_colsum_workspace_bytes(B*S, H, tile_rows) bytes (one cudaMemsetAsync on
 * `stream` before its kernel), so a call never depends on what an earlier
 * call left there. All calls share the one array: calls that can overlap on
 * the GPU (different streams, or different host threads without ordering)
 * race and give wrong results.
 */
#define DGR_COLSUM_NOALLOC_SCRATCH_BYTES (4u << 20)
dgr_status dgr_ordered_colsum_noalloc(const void *x, int32_t dtype, int64_t B, int64_t S, int64_t H,
                                      int64_t stride_b, int64_t stride_s, float *out, int32_t accumulate,
                                      int32_t tile_rows, void *stream);

/*
 * The status word of the no-alloc column sum's array on the current device,
 * as dgr_read_device_status() reads a workspace's: synchronises `stream`,
 * copies the word to *status (host pointer; DGR_OK when no device-side error
 * was recorded, DGR_ERR_TIMEOUT when a bounded wait ran out) and with
 * clear != 0 then zeroes it. The next dgr_ordered_colsum_noalloc() call
 * zeroes the word again, so read it after the call of interest and before the
 * next one (ordered on `stream`). Returns the read's own error, if any.
 */
dgr_status dgr_colsum_noalloc_read_status(int32_t clear, int32_t *status, void *stream);

/* ------------------------------------------------------------------------ */
/* 2. Ordered per-row dprob                                                  */
/* ------------------------------------------------------------------------ */
/*
 * cuDNN-frontend PR #521 ("grouped gemm dsrelu deterministic dprob"), commit
 * "deterministic dprob": dprob gets one FP32 slot per N-tile, so each
 * (token, tile_n) pair has exactly one writer; the slots are reduced in a
 * fixed order and the reduction accumulates into dprob.
 *
 *   dprob[m] = fold_j pw_W( dY[m][n] * Y[m][n] : n in tile j ),  W = tile_n,
 *   each product one fp32 multiply of the widened inputs, rounded on its own.
 *
 * dY, Y:    [M, N] row-major with leading dimensions ld_dy, ld_y (elements).
 * dprob:    [M] fp32; accumulate as for the column sum; N = 0 gives +0.0 /
 *           leaves dprob.
 * tile_n:   128 (the only width of the fused kernel).
 * slots:    NULL, or [M, ceil(N/tile_n)] fp32 receiving the tile partials
 *           (the low-level form of the page's class API).
 * Limits:   M <= 2^31 - 1, N <= 65536. Vector loads need 16-byte aligned rows.
 * ws:       dgr_rowdot_workspace_bytes() bytes (0: the fold stays on chip; ws
 *           may then be NULL).
 * dprob and slots must not overlap dY, Y or each other.
 */
size_t dgr_rowdot_workspace_bytes(int64_t M, int64_t N, int32_t tile_n);
dgr_status dgr_ordered_rowdot_dprob(const void *dY, const void *Y, int32_t dtype, int64_t M, int64_t N,
                                    int64_t ld_dy, int64_t ld_y, float *dprob, int32_t accumulate,
                                    int32_t tile_n, float *slots, void *ws, size_t ws_bytes,
                                    void *stream);

/* ------------------------------------------------------------------------ */
/* 3. Deterministic index_add                                                */
/* ------------------------------------------------------------------------ */
/*
 * Megatron-LM PR #7441 ("DSv4 --deterministic-mode"), Source 3: an
 * atomic-free index_add of gradient rows by a stable sort by destination and a
 * segmented sum, padding routed to a dummy row the caller drops.
 *
 *   key[i] = idx[i] if 0 <= idx[i] < R, else R (the dummy row);
 *   a stable sort orders the rows of each destination by original index;
 *   destination r's members, in that order, are cut into tiles of seg_tile
 *   and out[r][d] = out[r][d] + fold_tiles pw_{seg_tile}( src[i][d] ).
 *   Rows with no member are not touched.
 *
 * out:      [R+1, D] fp32, row stride ld_out (elements); row R is the dummy.
 * src:      [N, D] fp32, row stride ld_src. idx: [N] int32.
 * seg_tile: power of two, 1 .. 128 (128 canonical; 1 = plain sequential).
 * bad_count: NULL, or one device int32 that receives (overwrites) the number
 *           of idx entries outside [-1, R); those rows go to the dummy row.
 * Limits:   R + 1 <= 65536, N <= 2^31 - 1, D <= 4096. Rows of out and src
 *           need 16-byte alignment (ld_* and D multiples of 4).
 * ws:       dgr_index_add_workspace_bytes(N, R, D) bytes, zeroed once; it
 *           then serves every call with the same N and R and any D' <= D
 *           (D' = 0 included: the call then only counts bad indices). The
 *           first call records N and R in the workspace header; a later call
 *           with another N or R is refused on the device: it records
 *           DGR_ERR_INVALID_ARG in the status word and writes nothing (out and
 *           bad_count untouched); zero the workspace before using it for
 *           other sizes. Offsets read back from the workspace are clamped to
 *           their arrays, so a workspace left inconsistent (e.g. by a call that
 *           timed out) gives wrong sums, never an access out of bounds.
 * Residency: rows longer than 32 tiles of 128 are folded by blocks that wait,
 * bounded, for the tiles other blocks sum; the last launch takes one block
 * per SM usable at once (the device's, or a green context's partition), so
 * all are resident; the limits of the column sum's residency note apply.
 * out must not overlap src, idx, bad_count or ws.
 */
size_t dgr_index_add_workspace_bytes(int64_t N, int64_t R, int64_t D);
dgr_status dgr_det_index_add(float *out, int64_t R, int64_t D, int64_t ld_out, const float *src,
                             int64_t ld_src, const int32_t *idx, int64_t N, int32_t seg_tile,
                             int32_t *bad_count, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* 4. Split-K grouped weight gradient, accumulated into fp32 main_grad       */
/* ------------------------------------------------------------------------ */
/*
 * FlashInfer PR #8602 ("fuse the fp32 weight-gradient accumulate into
 * main_grad") and its follow-up #8924 ("Design and numerics"): out[e] gets
 * G_e^T X_e added; the deterministic form computes dW with a fixed split
 * order and then one RN32(out + dW); an empty group leaves out bitwise
 * unchanged. The 512-token k tile is the weight-gradient main stage.
 *
 *   for expert e (tokens offs[e] .. offs[e+1]-1), chunk c of chunk_tokens
 *   tokens from the expert's first token (the last chunk zero-filled):
 *     p_c[n][k] = sum over the chunk of G[t][n] * X[t][k] on the tensor cores,
 *                 from a fresh accumulator, K16 steps in ascending token order;
 *   dW = fold_c p_c (ascending, starting from p_0);
 *   main_grad[e][n][k] = main_grad[e][n][k] + dW[n][k]   (one rounding).
 * The last add is made in L2 by the bulk copy engine's tensor reduce-add,
 * one round-to-nearest-even binary32 add per element with subnormals kept;
 * every element has exactly one writer, so nothing depends on timing. (A NaN
 * result is a NaN; its payload is not specified.)
 *
 * G:        [T_total, N] bf16 row-major; X: [T_total, K] bf16 row-major.
 * d_offs:   [E+1] int64 DEVICE array, non-decreasing, d_offs[0] = 0,
 *           d_offs[E] = T_total (not read by the host: no synchronisation).
 * main_grad: [E, N, K] fp32, dense.
 * chunk_tokens: 512.
 * Limits:   N a multiple of 128, K a multiple of 256, E >= 1, T_total < 2^31,
 *           N, K <= 2^20, E * N < 2^31 (DGR_ERR_UNSUPPORTED otherwise).
 * Alignment: G, X 16-byte aligned; main_grad 32-byte aligned.
 * ws:       dgr_wgrad_workspace_bytes() bytes, zeroed once (status word).
 * main_grad must not overlap G, X, d_offs or ws.
 * T_total = 0 (every expert empty): nothing is launched and main_grad stays
 * as it is; G and X may then be null.
 */
size_t dgr_wgrad_workspace_bytes(int32_t E, int64_t N, int64_t K);
dgr_status dgr_grouped_wgrad_accumulate(const void *G, const void *X, const int64_t *d_offs, int32_t E,
                                        int64_t T_total, int64_t N, int64_t K, float *main_grad,
                                        int32_t chunk_tokens, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* 5. Grouped dbias: an ordered column sum per expert's rows                 */
/* ------------------------------------------------------------------------ */
/*
 * cuDNN-frontend PR #521, commit "Cover dbias": dbias contends across M-tiles,
 * so each (row block, column) gets one FP32 partial with a single writer and a
 * per-expert segment sum reduces the partials in a fixed order; the reduction
 * accumulates into dbias like the dprob one (commit "Address PR review").
 *
 *   expert e owns rows d_offs[e] .. d_offs[e+1]-1 of dY; its tiles are
 *   tile_rows consecutive rows counted from its first row (the last one
 *   ragged);
 *   dbias[e][h] = fold_j pw_W( dY[t][h] : t in tile j of expert e ),
 *   written (accumulate = 0) or added with one rounding (accumulate != 0);
 *   an expert with no rows gets +0.0 (overwrite) or is left unchanged.
 *
 * dY:       [T, H] bf16 or fp32 (dtype), row stride ld_dy (elements).
 * d_offs:   [E+1] int64 DEVICE array, non-decreasing, d_offs[0] = 0,
 *           d_offs[E] = T (never read by the host: no synchronisation). Offsets
 *           outside this contract are detected on the device: the call then
 *           writes nothing and records DGR_ERR_INVALID_ARG in the status word.
 * dbias:    [E, H] fp32, row stride ld_out (elements).
 * tile_rows: power of two 8 .. 128 (128 canonical).
 * Limits:   1 <= E <= 1024, T < 2^31, H <= 2^20. dY 16-byte aligned with H
 *           and ld_dy multiples of 16 bytes' worth of elements (8 bf16, 4 fp32):
 *           DGR_ERR_MISALIGNED otherwise.
 * ws:       dgr_dbias_workspace_bytes(T, H, E, tile_rows) bytes, zeroed once
 *           (status word, FP32 partials).
 * dbias must not overlap dY, d_offs or ws.
 */
size_t dgr_dbias_workspace_bytes(int64_t T, int64_t H, int32_t E, int32_t tile_rows);
dgr_status dgr_grouped_dbias(const void *dY, int32_t dtype, int64_t T, int64_t H, int64_t ld_dy,
                             const int64_t *d_offs, int32_t E, float *dbias, int64_t ld_out,
                             int32_t accumulate, int32_t tile_rows, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* 6. Canonical compact top-K                                                */
/* ------------------------------------------------------------------------ */
/*
 * Megatron-LM PR #7441, Source 1 and its fix _canonicalize_compact_topk: the
 * compact top-K returns each row's ids in a run-dependent slot order and
 * accumulates its softmax in that order; the ids are sorted per row with
 * padding last, the logits permuted alike and the softmax recomputed in that
 * order; rows that are all padding become 0 rather than NaN.
 *
 *   per row: slots sorted stably by id, ids < 0 (padding) after every id;
 *   out_ids[k] = ids[perm[k]], out_logits[k] = logits[perm[k]];
 *   over the n valid slots (they come first): m = max logit, d = RN(l - m),
 *   e = expf(d), Z = canonical sum of e in sorted order (tiles of 128,
 *   pairwise inside, ascending fold), probs[k] = RN(e_k / Z); padding slots
 *   and all-padding rows get +0.0.
 *
 * ids:      [R, K] int32, row stride ld_ids; logits: [R, K] fp32, ld_logits.
 * out_ids, out_logits, probs: [R, K], row stride ld_out; none may overlap an
 *           input or each other.
 * Limits:   1 <= K <= 256. No workspace: rows are independent.
 */
dgr_status dgr_topk_canonicalize(const int32_t *ids, int64_t ld_ids, const float *logits, int64_t ld_logits,
                                 int64_t R, int32_t K, int32_t *out_ids, float *out_logits, float *probs,
                                 int64_t ld_out, void *stream);

/* ------------------------------------------------------------------------ */
/* 7. Deterministic aux-loss scalar                                          */
/* ------------------------------------------------------------------------ */
/*
 * Megatron-LM PR #7441, Source 5: the fused router aux loss reduces its scalar
 * with a cross-block float atomicAdd; its gradient is the closed form
 * coeff*E/(topk*N^2)*tokens_per_expert[e], so the loss is that factor times
 * sum over t, e of probs[t][e] * tokens_per_expert[e]. Here:
 *
 *   x[t] = fold over expert tiles of pw_128( RN(probs[t][e] * tpe[e]) );
 *   S    = fold over token tiles of pw_128( x[t] );
 *   *d_out = RN(scale * S)        (N = 0: RN(scale * +0.0)).
 *
 * probs:    [N, E] fp32, row stride ld (elements). tokens_per_expert: [E]
 *           int32 DEVICE counts (exact in binary32 below 2^24).
 * scale:    the caller's factor, e.g. coeff * E / (topk * N^2).
 * d_out:    one DEVICE fp32 (overwritten).
 * Limits:   1 <= E <= 1024, N < 2^31.
 * ws:       dgr_aux_loss_workspace_bytes(N) bytes, zeroed once (a ticket and
 *           one FP32 partial per tile of 128 tokens).
 * d_out must not overlap probs, tokens_per_expert or ws.
 */
size_t dgr_aux_loss_workspace_bytes(int64_t N);
dgr_status dgr_aux_loss(const float *probs, int64_t N, int32_t E, int64_t ld, const int32_t *d_tokens_per_expert,
                        float scale, float *d_out, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* 8. dprob fused into its grouped dsReLU GEMM                               */
/* ------------------------------------------------------------------------ */
/*
 * cuDNN-frontend PR #521 ("grouped gemm dsrelu deterministic dprob"): the
 * backward kernel recomputes the grouped GEMM, reuses relu(C)^2 for dprob,
 * and makes dprob deterministic with one partial per (token, N-tile), a single
 * writer each, reduced in a fixed order and accumulated into dprob. For the
 * tokens of expert e (rows d_offs[e] .. d_offs[e+1]-1):
 *
 *   C[m][n] = sum_k A[m][k] B[e][k][n] on the tensor cores (K16 steps over k
 *             ascending, from a fresh accumulator; fp32);
 *   leaf    = RN(fp32(dY[m][n]) * RN(r * r)), r = max(C[m][n], 0);
 *   dprob[m] = fold over N-tiles of 128 of pw_128(leaves), written
 *             (accumulate = 0) or added with one rounding.
 *
 * C is never written. A: [T, K] bf16 row-major; B: [E, K, N] bf16 row-major;
 * dY: [T, N] bf16 row-major; dprob: [T] fp32; d_offs: [E+1] int64 DEVICE,
 * non-decreasing, d_offs[0] = 0, d_offs[E] = T (checked on the device: the call
 * then writes nothing and records DGR_ERR_INVALID_ARG in the status word).
 * Limits:   K a multiple of 64, N a multiple of 256, 1 <= E <= 1024, T < 2^31.
 * Alignment: A, B, dY 16-byte aligned.
 * ws:       dgr_dsrelu_dprob_workspace_bytes(T, N) bytes, zeroed once (status
 *           word, one FP32 partial per token and N-tile).
 * dprob must not overlap A, B, dY, d_offs or ws.
 * T = 0 (every expert empty): nothing is launched; A, B, dY, dprob and ws may
 * then be null.
 */
size_t dgr_dsrelu_dprob_workspace_bytes(int64_t T, int64_t N);
dgr_status dgr_dsrelu_dprob(const void *A, const void *B, const int64_t *d_offs, int32_t E, int64_t T, int64_t K,
                            int64_t N, const void *dY, float *dprob, int32_t accumulate, void *ws, size_t ws_bytes,
                            void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DGR_H */
