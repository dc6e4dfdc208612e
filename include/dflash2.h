/*
 * dflash2.h — C ABI of the GB300 (sm_103a) DFlash2 draft-proposal hot path.
 *
 * The method is the one of sglang PR "[Spec] DFlash2: local convolution +
 * candidate selector" (a block-causal grouped dynamic conv, unary candidate
 * logits with a top-K, and a low-rank selector lattice walked slot by slot),
 * plus the draft-to-target id remap of vLLM PR "DSpark padded-vocab drafts no
 * longer wrongly demand a d2t table" (map_draft_to_target).
 *
 * General rules for every entry point
 *   - Pointers named as device pointers must point to device memory that the
 *     caller allocated and keeps alive until the work queued on `stream`
 *     completes.  The library allocates nothing, keeps no per-call state,
 *     never synchronises and never falls back to the CPU.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *     work is queued on it asynchronously, in call order.
 *   - Arguments are validated on the host before anything is queued; a bad
 *     argument returns a non-OK status and queues nothing.
 *   - `err_word` (device int32, caller-owned, may be NULL where noted) is
 *     OR-ed with DFLASH2_DEVERR_* bits by the kernels when they meet data
 *     they cannot process (for example an id outside its table); the kernels
 *     then write a defined value (id 0, a zero table row) and carry on.  The
 *     caller clears it and reads it back when it synchronises.
 *   - dtype is DFLASH2_F32 or DFLASH2_BF16 and applies to every floating
 *     tensor of the call unless stated otherwise.  Ids are int64.
 *   - The kernels are built for sm_103a only; on any other device every
 *     compute entry point returns DFLASH2_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef DFLASH2_H
#define DFLASH2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH2_ABI_VERSION 9

typedef enum {
    DFLASH2_OK = 0,
    DFLASH2_ERR_INVALID_ARG = 1,        /* a null pointer, a size out of range */
    DFLASH2_ERR_UNSUPPORTED_DTYPE = 2,  /* dtype not fp32/bf16 (e.g. a quantised head) */
    DFLASH2_ERR_MISALIGNED = 3,         /* a pointer or stride breaks an alignment rule */
    DFLASH2_ERR_WORKSPACE = 4,          /* workspace null or smaller than the minimum */
    DFLASH2_ERR_CUDA = 5,               /* a CUDA runtime call failed (launch, attribute) */
    DFLASH2_ERR_UNSUPPORTED_DEVICE = 6  /* current device is not sm_103 */
} dflash2_status;

typedef enum { DFLASH2_F32 = 0, DFLASH2_BF16 = 1 } dflash2_dtype;

/* Bits OR-ed into *err_word by the kernels. */
#define DFLASH2_DEVERR_ID_RANGE 0x1  /* an id outside [0, rows of its table) */
#define DFLASH2_DEVERR_TIMEOUT 0x2   /* a bounded pipeline wait gave up; outputs invalid */
#define DFLASH2_DEVERR_SHORT 0x4     /* fewer than K selectable vocab entries */
/* Informational (not an error): a top-K row overflowed its candidate list and
 * was recomputed exactly on CUDA cores. */
#define DFLASH2_DEVINFO_TOPK_FALLBACK 0x100

/* Human-readable name of a status code (static storage). */
const char *dflash2_status_string(int32_t status);

/* DFLASH2_ABI_VERSION of the loaded library. */
int32_t dflash2_abi_version(void);

/*
 * Block-causal grouped dynamic depthwise convolution.
 * sglang DFlash2 PR, _grouped_conv and DFlashGroupedConv: hidden is split into
 * groups of `group_size` channels; tap t of token i uses the coefficient
 * base[t, c] + delta[i, t, c / group_size] on x[i - t, c], and is zeroed unless
 * the in-block position i mod block_size is at least t:
 *
 *   out[i, c] = sum_{t < taps, (i mod block_size) >= t}
 *               (base[t, c] + delta[i, t, c / group_size]) * x[i - t, c]
 *
 * x, out      device, [n_tokens, hidden] row-major, token-major; each request's
 *             block of block_size rows is contiguous (the last block may be short).
 * base        device, [taps, hidden] (one side of the module's [2, taps, hidden]).
 * delta       device; row i starts at delta + i * delta_row_stride elements and
 *             holds [taps, hidden / group_size].  delta_row_stride >= taps * groups
 *             lets side 0 of a [n, 2, taps, groups] projection be read in place.
 * Arithmetic: fp32 (coefficient formed in fp32, fp32 multiply-add, taps in
 *             order 0..taps-1); out is rounded to dtype.
 * Errors:     hidden % group_size != 0, taps < 1, block_size < 1, n_tokens < 0,
 *             delta_row_stride < taps * groups -> INVALID_ARG.  n_tokens == 0
 *             queues nothing.  out must not overlap x.
 * The fast path wants x, base and out 16-byte aligned and group_size a multiple
 * of 8 (bf16) or 4 (fp32); other layouts take a scalar path.
 */
dflash2_status dflash2_grouped_conv(const void *x, const void *base, const void *delta,
                                    int64_t delta_row_stride, void *out, int64_t n_tokens,
                                    int32_t hidden, int32_t group_size, int32_t taps,
                                    int32_t block_size, int32_t dtype, void *stream);

/*
 * Unary candidates: lm_head GEMM, output transform, padded-vocab mask, top-K.
 * sglang DFlash2 PR, DFlash2DraftModel.compute_candidates / _transform_unary_logits
 * / _radix_topk and _selector_lattice (the rows are the flattened
 * [batch, slots] proposals); vLLM DSpark padded-vocab review (mask
 * [target_vocab, draft_vocab) before top-k).
 *
 *   z[m, v] = sum_j h[m, j] * lm_head[v, j]
 *   u[m, v] = cap * tanh(mult * z / cap)  if cap > 0,  mult * z  otherwise
 *   u[m, v] = -inf                        for v >= target_vocab
 *   cand_ids[m, :], cand_u[m, :] = the top_k (u, v) of row m, ordered by u
 *                                  descending, equal u by smaller v
 *
 * h           device, [rows, hidden] row-major (proposal positions only).
 * lm_head     device, [draft_vocab, hidden] row-major (nn.Linear weight layout).
 * cand_ids    device int64 [rows, top_k];  cand_u device float [rows, top_k].
 * workspace   device, ws_bytes >= dflash2_unary_topk_workspace_min(...);
 *             dflash2_unary_topk_workspace_size(...) is the recommended size.
 *             Its contents need no initialisation and are clobbered.  fp32 needs
 *             none (min 0); with the recommended size (8-byte aligned) a few
 *             rows' vocab is split over CTAs and the lists merged exactly.
 * err_word    device int32, may be NULL.
 * Arithmetic: bf16 -> tcgen05 tensor-core GEMM with fp32 accumulation; fp32 ->
 *             fp32 FMA on CUDA cores (no TF32).  The transform runs in fp32
 *             (tanhf), and selection compares the fp32 u.
 * Errors:     INVALID_ARG for rows outside [0, 2^31), hidden outside [1, 32768],
 *             draft_vocab outside [1, 2^31), target_vocab < 1, top_k outside
 *             [1, 128] or above either vocab size, cap negative or NaN, or a null
 *             pointer; UNSUPPORTED_DTYPE for a dtype other than f32 / bf16;
 *             MISALIGNED for cand_ids not 8-byte or cand_u not 4-byte aligned, and
 *             for bf16 when hidden % 8 != 0, h or lm_head is not 16-byte aligned
 *             or the workspace is not 256-byte aligned; WORKSPACE for a bf16
 *             workspace below the minimum.  rows == 0 queues nothing.
 * Device:     a row whose candidate list outgrows the workspace is recomputed
 *             exactly on CUDA cores and flagged DFLASH2_DEVINFO_TOPK_FALLBACK (not
 *             an error); fewer than top_k valid entries set DFLASH2_DEVERR_SHORT.
 */
size_t dflash2_unary_topk_workspace_size(int64_t rows, int64_t draft_vocab, int32_t top_k,
                                         int32_t dtype);
size_t dflash2_unary_topk_workspace_min(int64_t rows, int64_t draft_vocab, int32_t top_k,
                                        int32_t dtype);
/*
 * Kernels one dflash2_unary_topk call with these shapes queues on the current
 * device: for fp32 1, or 2 when the recommended workspace splits the vocab
 * over CTAs (chunks, then dflash2_topk_merge; counted for target_vocab >=
 * draft_vocab); for bf16 either 2 (one cooperative launch of the pilot
 * tiles, the thresholds and the filter tiles, then the final top-K) or 3 / 4
 * (pilot pass, pilot select, filter pass unless the pilot covers the vocab,
 * final top-K); 0 for rows == 0.  Host arithmetic only, nothing is queued;
 * -1 for a dtype, rows, draft_vocab or top_k that dflash2_unary_topk rejects, or
 * when no device is usable.  (dflash2_unary_topk also queues a memset of
 * 8 bytes before the cooperative launch.)
 */
int32_t dflash2_unary_topk_launches(int64_t rows, int64_t draft_vocab, int32_t top_k, float mult,
                                    int32_t dtype);
dflash2_status dflash2_unary_topk(const void *h, const void *lm_head, int64_t rows,
                                  int32_t hidden, int64_t draft_vocab, int64_t target_vocab,
                                  float mult, float cap, int32_t top_k, int32_t dtype,
                                  int64_t *cand_ids, float *cand_u, void *workspace,
                                  size_t ws_bytes, int32_t *err_word, void *stream);

/*
 * FP8 (E4M3) lm_head: the unary candidates of an FP8 head checkpoint.  The
 * sglang DFlash2 PR lets a quantized lm_head fall back to its eager path;
 * this computes the same candidates from the quantized head on the tensor
 * cores (tcgen05.mma kind::f8f6f4).  W8A8 with per-row scales:
 *
 *   activation codes, per row m of h (dflash2_quantize_rows_e4m3):
 *     amax = max_j |h[m, j]|, inv = 448 / amax, d[m] = amax / 448 (fp32),
 *     q_h[m, j] = E4M3(h[m, j] * inv)   (fp32 product, round to nearest even,
 *     saturating at +-448; a row of zeros: codes 0, d = 1)
 *   z[m, v] = d[m] * w_scale[v] * sum_j dec(q_h[m, j]) * dec(lm_head_q[v, j])
 *   then the transform, the padded-vocab mask and the top-K of
 *   dflash2_unary_topk.
 *
 * E4M3 is the OCP 8-bit "e4m3fn" format (bias 7, 3 mantissa bits, max 448,
 * no infinities, 0x7F / 0xFF NaN).
 *
 * dflash2_quantize_rows_e4m3: x device [rows, cols] (dtype f32 or bf16) ->
 *   q device uint8 [rows, cols], scale device float [rows].
 *   Errors: dtype -> UNSUPPORTED_DTYPE; rows outside [0, 2^31), cols < 1 or a
 *   null pointer -> INVALID_ARG; x or scale misaligned for its type ->
 *   MISALIGNED.  rows == 0 queues nothing.
 * dflash2_unary_topk_fp8: h device [rows, hidden] (h_dtype f32 or bf16);
 *   lm_head_q device uint8 [draft_vocab, hidden] E4M3 codes, 16-byte aligned;
 *   w_scale device float [draft_vocab]; the other arguments as for
 *   dflash2_unary_topk.  hidden % 16 == 0 (the codes' rows are TMA rows).
 *   workspace device, 256-byte aligned, ws_bytes >=
 *   dflash2_unary_topk_fp8_workspace_size(rows, hidden, draft_vocab, top_k):
 *   the activation codes and scales, then a dflash2_unary_topk workspace.
 *   Queues the quantization kernel and then what dflash2_unary_topk_launches
 *   reports for bf16.  Errors as for dflash2_unary_topk, plus MISALIGNED for
 *   hidden % 16 != 0 or lm_head_q not 16-byte aligned.
 * Arithmetic: exact products of codes summed in fp32 in the tensor cores,
 *   then z = acc * (d[m] * w_scale[v]) in fp32.
 */
dflash2_status dflash2_quantize_rows_e4m3(const void *x, int64_t rows, int32_t cols, int32_t dtype,
                                          uint8_t *q, float *scale, void *stream);
size_t dflash2_unary_topk_fp8_workspace_size(int64_t rows, int32_t hidden, int64_t draft_vocab,
                                             int32_t top_k);
dflash2_status dflash2_unary_topk_fp8(const void *h, int32_t h_dtype, const uint8_t *lm_head_q,
                                      const float *w_scale, int64_t rows, int32_t hidden,
                                      int64_t draft_vocab, int64_t target_vocab, float mult,
                                      float cap, int32_t top_k, int64_t *cand_ids, float *cand_u,
                                      void *workspace, size_t ws_bytes, int32_t *err_word,
                                      void *stream);

/*
 * NVFP4 lm_head: the unary candidates of an NVFP4 head checkpoint (the vLLM
 * DSpark review's padded-vocab draft ships one; the sglang DFlash2 PR lets a
 * quantized head fall back to its eager path).  W4A4 on the block-scaled
 * tensor cores (tcgen05.mma kind::mxf4nvf4, scale_vec::4X, CTA pairs):
 *
 *   E2M1 element: sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
 *     0, 0.5, 1, 1.5, 2, 3, 4, 6.  Two codes per byte, element 2i in the low
 *     nibble.  Every 16 consecutive elements along hidden share one E4M3
 *     scale (non-negative).
 *   activations, per row m of h (dflash2_quantize_rows_nvfp4), in fp32:
 *     amax = max_j |h[m, j]|, enc = 2688 / amax, g_h[m] = amax / 2688
 *     (2688 = 6 * 448; a row of zeros: enc = g_h = 1);
 *     block b: a_b = max |h| over its 16 elements, s_b = E4M3((a_b / 6) * enc);
 *     codes E2M1(h[m, j] * (enc / dec(s_b))) (round to nearest even,
 *     saturating at 6), all 0 when s_b is 0.
 *   weights: codes lm_head_q, block scales, one fp32 w_global, quantized
 *     the same way with the amax of the whole tensor (a checkpoint's format);
 *     the block scales are handed over as scale tiles (below).
 *   z[m, v] = g_h[m] * w_global * sum_b dec(s_h[m, b]) * dec(w_scales[v, b])
 *             * sum_{j in b} dec(q_h[m, j]) * dec(lm_head_q[v, j])
 *   then the transform, the padded-vocab mask and the top-K of
 *   dflash2_unary_topk.
 *
 * dflash2_quantize_rows_nvfp4: x device [rows, cols] (dtype f32 or bf16),
 *   cols % 16 == 0 -> codes device uint8 [rows, cols / 2] (8-byte aligned),
 *   scales device uint8 [rows, cols / 16], g device float [rows].
 *   Errors: dtype -> UNSUPPORTED_DTYPE; rows outside [0, 2^31), cols < 1 or
 *   not a multiple of 16, or a null pointer -> INVALID_ARG; x, codes or g
 *   misaligned -> MISALIGNED.  rows == 0 queues nothing.
 * dflash2_nvfp4_tile_scales: scales device uint8 [rows, hidden / 16]
 *   (row-major, 4-byte aligned), hidden % 64 == 0 -> tiles device, 16-byte
 *   aligned, dflash2_nvfp4_scale_tiles_size(rows, hidden) bytes, fully
 *   written.  The layout the block-scaled GEMM copies from: rows in blocks of
 *   128, a row's scales in cells of 4 bytes (64 elements), cells per row
 *   rounded up to nw8 = a multiple of 8; tile (rb, w) is 512 bytes at
 *   (rb * nw8 + w) * 512, row rb * 128 + l + 32 j (l < 32, j < 4) with its
 *   cell w at byte l * 16 + j * 4; everything else zero.  Call once per
 *   checkpoint.  Errors: INVALID_ARG (shape, null), MISALIGNED.
 * dflash2_unary_topk_nvfp4: h device [rows, hidden] (h_dtype f32 or bf16);
 *   lm_head_q device uint8 [draft_vocab, hidden / 2], 16-byte aligned;
 *   w_scale_tiles device: the weights' block scales as written by
 *   dflash2_nvfp4_tile_scales, 16-byte aligned;
 *   w_global > 0 and finite; hidden % 64 == 0; the other arguments as for
 *   dflash2_unary_topk.  workspace device, 256-byte aligned, ws_bytes >=
 *   dflash2_unary_topk_nvfp4_workspace_size(rows, hidden, draft_vocab,
 *   top_k): the activation codes, scales and g, then a dflash2_unary_topk
 *   workspace.  Queues the quantization and scale-tiling kernels, then the
 *   pair GEMM (fused with the select, or pilot, select and filter passes)
 *   and the final top-K.
 *   Errors as for dflash2_unary_topk, plus INVALID_ARG for hidden % 64 != 0 or
 *   a bad w_global, MISALIGNED for lm_head_q or w_scale_tiles.
 * Arithmetic: exact products of codes, summed per 16-element block and
 *   scaled by the two block scales in the tensor cores (fp32 accumulation),
 *   then z = acc * (g_h[m] * w_global) in fp32.
 */
dflash2_status dflash2_quantize_rows_nvfp4(const void *x, int64_t rows, int32_t cols,
                                           int32_t dtype, uint8_t *codes, uint8_t *scales,
                                           float *g, void *stream);
size_t dflash2_nvfp4_scale_tiles_size(int64_t rows, int32_t hidden);
dflash2_status dflash2_nvfp4_tile_scales(const uint8_t *scales, int64_t rows, int32_t hidden,
                                         uint8_t *tiles, void *stream);
size_t dflash2_unary_topk_nvfp4_workspace_size(int64_t rows, int32_t hidden, int64_t draft_vocab,
                                               int32_t top_k);
dflash2_status dflash2_unary_topk_nvfp4(const void *h, int32_t h_dtype, const uint8_t *lm_head_q,
                                        const uint8_t *w_scale_tiles, float w_global, int64_t rows,
                                        int32_t hidden, int64_t draft_vocab, int64_t target_vocab,
                                        float mult, float cap, int32_t top_k, int64_t *cand_ids,
                                        float *cand_u, void *workspace, size_t ws_bytes,
                                        int32_t *err_word, void *stream);

/*
 * Selector lattice and walk.
 * sglang DFlash2 PR: the PR body's edge formula
 *   edge(p -> c) = < A[p] (elementwise *) project(h), B[c] > + unary[c]
 * and _selector_walk_kernel / stage_sampling_params.  project(h) = h . proj^T
 * (proj is an nn.Linear(hidden, rank) weight).  Per request b, slot s:
 *   p      = anchor_ids[b] at s = 0, else cand_ids[b, s-1, previous]
 *   e[k]   = sum_j A[p, j] * g[b, s, j] * B[cand_ids[b, s, k], j] + cand_u[b, s, k]
 *   greedy[b] != 0:  index = smallest k with e[k] == max e;  q = one-hot(index)
 *   otherwise:       T = max(temperatures[b], 1e-5);  q = softmax(e / T);
 *                    index = min(#{k : uniforms[b, s] >= cumsum(q)[k]}, top_k - 1)
 *   tokens[b, s] = cand_ids[b, s, index];  previous = index
 *
 * h             device, [batch * slots, hidden] (same rows as unary_topk's h).
 * proj          device, [rank, hidden].
 * A, B          device, [table_rows, rank], indexed by draft ids.
 * anchor_ids    device int64 [batch]: the verified token at block position 0.
 * cand_ids      device int64 [batch, slots, top_k]; cand_u device float, same shape
 *               (the outputs of dflash2_unary_topk).
 * temperatures  device float [batch]; greedy device uint8 [batch];
 * uniforms      device float [batch, slots] in [0, 1).
 * tokens        device int64 [batch, slots]; q device float [batch, slots, top_k].
 * path_scores   device float [batch, slots, top_k] or NULL: the edges e[k] of the
 *               lattice row the walk actually read at each slot.
 * workspace     device, 16-byte aligned, ws_bytes >=
 *               dflash2_selector_walk_workspace_size(batch, slots, hidden, rank,
 *               top_k, dtype): the projection partials and, for top_k <= 32, the
 *               lattice of every request (edges, row statistics, draws).
 * Arithmetic: g in fp32 (bf16: tcgen05 GEMM; fp32: CUDA-core FMA), edges,
 *             softmax (expf) and the running sum in fp32.
 * Errors:     top_k < 1 or > 128, rank < 1 or > 256, rank % 8 != 0 (bf16) or
 *             % 4 != 0 (fp32), batch/slots < 0 -> INVALID_ARG.  An anchor or
 *             candidate id outside [0, table_rows) sets DFLASH2_DEVERR_ID_RANGE
 *             and uses a zero table row.
 */
size_t dflash2_selector_walk_workspace_size(int32_t batch, int32_t slots, int32_t hidden,
                                            int32_t rank, int32_t top_k, int32_t dtype);
dflash2_status dflash2_selector_walk(const void *h, const void *proj, const void *A,
                                     const void *B, int64_t table_rows,
                                     const int64_t *anchor_ids, const int64_t *cand_ids,
                                     const float *cand_u, const float *temperatures,
                                     const uint8_t *greedy, const float *uniforms,
                                     int32_t batch, int32_t slots, int32_t hidden,
                                     int32_t rank, int32_t top_k, int32_t dtype,
                                     int64_t *tokens, float *q, float *path_scores,
                                     void *workspace, size_t ws_bytes, int32_t *err_word,
                                     void *stream);

/*
 * The selector walk in two calls, so that the projection (which needs only h)
 * can run on another stream while the unary candidates are computed.  The
 * sglang DFlash2 PR computes project(h) inside build_lattice; splitting it changes no
 * arithmetic: the two calls together give exactly what dflash2_selector_walk
 * gives for the same arguments.
 *
 * dflash2_selector_project  step a5 alone: writes the fp32 partials of
 *   g = h . proj^T to the start of `workspace` (the same bytes
 *   dflash2_selector_walk uses for them).  h, proj, batch, slots, hidden,
 *   rank, dtype as for dflash2_selector_walk; top_k only sizes the workspace.
 * dflash2_selector_walk_projected  the edges and the walk from the partials
 *   a dflash2_selector_project call with the same batch, slots, hidden, rank,
 *   top_k and dtype left in `workspace`; the other arguments as for
 *   dflash2_selector_walk.  The caller orders the two calls (same stream, or
 *   an event); nothing checks that the partials are there.
 * Both: workspace device, 16-byte aligned, ws_bytes >=
 *   dflash2_selector_walk_workspace_size(batch, slots, hidden, rank, top_k,
 *   dtype); the same errors as dflash2_selector_walk for the arguments they
 *   take.
 */
dflash2_status dflash2_selector_project(const void *h, const void *proj, int32_t batch,
                                        int32_t slots, int32_t hidden, int32_t rank,
                                        int32_t top_k, int32_t dtype, void *workspace,
                                        size_t ws_bytes, int32_t *err_word, void *stream);
dflash2_status dflash2_selector_walk_projected(const void *A, const void *B, int64_t table_rows,
                                               const int64_t *anchor_ids,
                                               const int64_t *cand_ids, const float *cand_u,
                                               const float *temperatures, const uint8_t *greedy,
                                               const float *uniforms, int32_t batch,
                                               int32_t slots, int32_t hidden, int32_t rank,
                                               int32_t top_k, int32_t dtype, int64_t *tokens,
                                               float *q, float *path_scores, void *workspace,
                                               size_t ws_bytes, int32_t *err_word,
                                               void *stream);

/*
 * Selector walk without a workspace argument.  The DFlash2 PR has no counterpart:
 * this is a library convenience for callers that cannot provide device
 * memory at call time, such as serving loops whose device memory belongs to
 * another allocator (a caching allocator that reserved its pool up front and
 * must not be bypassed), or latency-critical paths that must never call
 * cudaMalloc / cudaFree, which can synchronise the whole device.
 *
 * Same arguments, meaning and result as dflash2_selector_walk, minus
 * workspace and ws_bytes.  It allocates nothing: its scratch is a fixed
 * 4 MiB (4194304-byte) array in the library's device memory, held by every
 * GPU that loads the library until the process exits.
 *   - The arguments are checked first, as dflash2_selector_walk checks them
 *     (an invalid shape returns INVALID_ARG or UNSUPPORTED_DTYPE; batch or
 *     slots 0 queues nothing and touches no device state).  Then a call whose
 *     scratch need (dflash2_selector_walk_workspace_size of its shapes: the
 *     projection partials, plus the lattice when top_k <= 32) exceeds 4 MiB
 *     returns DFLASH2_ERR_WORKSPACE and queues nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the
 *     life of the process; make that first call before any stream capture.
 *     The kept address assumes the device's primary context is not reset
 *     (cudaDeviceReset) while the library is loaded.
 *   - Every call, on every stream, shares the one array and overwrites what
 *     the previous call left there (nothing in it needs to start at zero).
 *     Calls whose work overlaps on the GPU, on different streams or from
 *     different threads, race on it: serialise them.
 */
dflash2_status dflash2_selector_walk_noalloc(const void *h, const void *proj, const void *A,
                                             const void *B, int64_t table_rows,
                                             const int64_t *anchor_ids, const int64_t *cand_ids,
                                             const float *cand_u, const float *temperatures,
                                             const uint8_t *greedy, const float *uniforms,
                                             int32_t batch, int32_t slots, int32_t hidden,
                                             int32_t rank, int32_t top_k, int32_t dtype,
                                             int64_t *tokens, float *q, float *path_scores,
                                             int32_t *err_word, void *stream);

/*
 * Grouped-conv prepare: the kernel projection, then the input-side conv.
 * sglang DFlash2 PR, DFlashGroupedConv.prepare: one bias-free linear map
 * kernel_projection = Linear(hidden, 2 * taps * groups) gives each token the
 * dynamic coefficients of both convolutions of a wrapped sublayer,
 *
 *   coef[i, r] = sum_j x[i, j] * w_kp[r, j],   r = (side * taps + t) * groups + g,
 *
 * stored in dtype (bf16: fp32 accumulation on the tensor cores, rounded to
 * nearest-even once); then out = the grouped conv of x with base side 0 and
 * coefficient side 0 (dflash2_grouped_conv, delta read in place with row
 * stride 2 * taps * groups).  Side 1 stays in coef for dflash2_conv_finish.
 *
 * x, out   device, [n_tokens, hidden] as for dflash2_grouped_conv.
 * w_kp     device, [2 * taps * groups, hidden] (nn.Linear weight layout).
 * base2    device, base_kernel [2, taps, hidden].
 * coef     device, [n_tokens, 2, taps, groups], written (caller-owned).
 * err_word device int32 or NULL; a projection wait that gives up sets
 *          DFLASH2_DEVERR_TIMEOUT.
 * Errors:  as dflash2_grouped_conv; bf16 also needs hidden % 8 == 0 and x,
 *          w_kp 16-byte aligned (tensor-memory-access copies) -> MISALIGNED.
 *          n_tokens == 0 queues nothing.
 */
dflash2_status dflash2_conv_prepare(const void *x, const void *w_kp, const void *base2,
                                    int64_t n_tokens, int32_t hidden, int32_t group_size,
                                    int32_t taps, int32_t block_size, int32_t dtype, void *out,
                                    void *coef, int32_t *err_word, void *stream);

/*
 * Grouped-conv finish: the output-side conv.
 * sglang DFlash2 PR, DFlashGroupedConv.finish: the sublayer's output y is
 * convolved with base side 1 and coefficient side 1 of the coef that
 * dflash2_conv_prepare wrote for the same tokens.  Arguments and errors as for
 * dflash2_grouped_conv; base2 and coef as for dflash2_conv_prepare.
 */
dflash2_status dflash2_conv_finish(const void *y, const void *base2, const void *coef,
                                   int64_t n_tokens, int32_t hidden, int32_t group_size,
                                   int32_t taps, int32_t block_size, int32_t dtype, void *out,
                                   void *stream);

/*
 * Lossless verification of a proposed block (speculative sampling).
 * The consumer of the walk's q; the pages do not print it, so this is the
 * standard rule of Leviathan et al. ("Fast inference from transformers via
 * speculative decoding", 2023) and Chen et al. ("Accelerating large language
 * model decoding with speculative sampling", 2023).  For request b, with
 * T' = max(T_b, 1e-5) as the walk clamps and p_s = softmax(logits[b, s] / T'):
 *
 *   slots s = 0 .. slots-1 in order, x = draft[b, s], k its candidate index:
 *     greedy row:  accept iff x == argmax_y logits[b, s, y] (smallest y on ties)
 *     sampled row: accept iff uniforms[b, s] * q[b, s, k] < p_s(x)
 *   first rejection at s: emit one token and stop;
 *     greedy: the argmax; sampled: a draw from max(0, p_s - qt) (qt = q on the
 *     slot's candidate ids, 0 elsewhere) by inverse CDF with u = uniforms[b, slots]
 *   no rejection: the bonus token from position `slots` (argmax, or a draw from
 *     p_slots with the same u).
 *
 * target_logits device, [batch, slots + 1, vocab] (dtype), the target model's
 *               logits at the block's positions.
 * draft, cand   device int64 [batch, slots] and [batch, slots, top_k]: TARGET ids
 *               (map the walk's tokens and candidates with dflash2_d2t_remap).
 * q             device f32 [batch, slots, top_k] (the walk's q).
 * uniforms      device f32 [batch, slots + 1] in [0, 1).
 * temperatures, greedy  as for dflash2_selector_walk.
 * accept_len    device int64 [batch]: accepted drafts (0 .. slots).
 * out_tokens    device int64 [batch, slots + 1]: the accepted drafts, the
 *               emitted token, then -1.
 * workspace     device, >= dflash2_verify_workspace_size(batch, slots, vocab)
 *               bytes, 16-byte aligned (per-chunk softmax partials).
 * Arithmetic: fp32; p = 2^(logit * log2(e) / T' - m) / Z with the hardware
 *   base-2 exponential (PTX ex2.approx.ftz.f32; the change of base is exact in
 *   real arithmetic, and the approximation is within the tolerance the
 *   near-tie rule allows); fixed reduction orders, so results are
 *   deterministic.
 * Errors: slots > 64, top_k outside [1, 128], vocab outside [1, 2^20] ->
 *   INVALID_ARG.  A draft that is not among its slot's candidates, or an id
 *   outside [0, vocab), sets DFLASH2_DEVERR_ID_RANGE and leaves that request's
 *   accept_len 0 and out_tokens -1.
 */
size_t dflash2_verify_workspace_size(int32_t batch, int32_t slots, int64_t vocab);
dflash2_status dflash2_verify(const void *target_logits, int64_t vocab,
                              const float *temperatures, const uint8_t *greedy,
                              const int64_t *draft, const int64_t *cand, const float *q,
                              const float *uniforms, int32_t batch, int32_t slots,
                              int32_t top_k, int32_t dtype, int64_t *accept_len,
                              int64_t *out_tokens, void *workspace, size_t ws_bytes,
                              int32_t *err_word, void *stream);

/*
 * Counter-based uniforms for the walk.
 * sglang DFlash2 PR, _SelectorDraftSampler: the uniforms of the sampled rows
 * are drawn inside the captured CUDA graph from a Philox generator whose state
 * advances at every replay (and the PR's risk list warns that a replay reusing
 * the sequence would break the sampling).  The generator is Philox4x64-10
 * (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
 *
 *   out[i] = (word[i % 4] >> 40) * 2^-24,
 *   word = Philox4x64_10(counter = (base + i / 4, 0, 0, 0), key = (seed, 0)),
 *
 * so out[i] lies in [0, 1) on the 2^-24 grid.
 *
 * counter == NULL: base = offset; any n >= 0.
 * counter != NULL: device uint64, read and advanced on the device:
 *                  base = *counter + offset, then *counter += ceil(n / 4).
 *                  A graph that captures the call draws a fresh sequence at
 *                  every replay.  n <= 2^24.  Calls that share a counter must be
 *                  ordered (one stream, or events).
 * out:             device float32 [n], 4-byte aligned (16-byte aligned stores
 *                  four at a time).
 * Errors: n < 0, out == NULL, or n > 2^24 with a counter -> INVALID_ARG;
 *         misaligned out or counter -> MISALIGNED.  n == 0 queues nothing and
 *         leaves the counter as it is.
 */
dflash2_status dflash2_philox_uniforms(uint64_t seed, uint64_t offset, uint64_t *counter,
                                       int64_t n, float *out, void *stream);

/*
 * Exact merge of vocab-sharded top-K lists (the one exchange of a
 * vocab-sharded unary top-K: each GPU runs dflash2_unary_topk over its slice
 * of lm_head rows, the [rows, k_in] lists are all-gathered, and every rank
 * merges them).  The sglang DFlash2 PR computes the candidates over the whole
 * vocab on one GPU; this splits the same computation.  The logits of a vocab
 * row do not depend on the slice that computes them, so the merge gives
 * exactly the unsharded dflash2_unary_topk result:
 *
 *   out[r, :] = the k_out largest (u, id_offsets[s] + ids[s, r, j]) over all
 *               shards s and j, ordered by u descending, equal u by smaller id
 *
 * ids         device int64 [shards, rows, k_in]: shard-local vocab ids.
 * u           device float [shards, rows, k_in]; u = -inf or NaN marks an
 *             absent entry (a shard with fewer than k_in selectable ids pads
 *             its list so, as dflash2_unary_topk does).  No order is assumed.
 * id_offsets  HOST int64 [shards]: the first global vocab id of each shard,
 *             in [0, 2^31).
 * out_ids     device int64 [rows, k_out]; out_u device float [rows, k_out].
 * Errors:     shards outside [1, 64], k_in < 1, k_out outside [1, 128],
 *             shards * k_in > 4096, rows outside [0, 2^31), an offset out of
 *             range or a null pointer -> INVALID_ARG; ids not 8-byte or u not
 *             4-byte aligned -> MISALIGNED.  rows == 0 queues nothing.
 * Device:     fewer than k_out present entries fill the rest with id 0 and
 *             -inf and set DFLASH2_DEVERR_SHORT; a global id outside
 *             [0, 2^32 - 1) is dropped and sets DFLASH2_DEVERR_ID_RANGE.
 */
dflash2_status dflash2_topk_merge(const int64_t *ids, const float *u, const int64_t *id_offsets,
                                  int32_t shards, int64_t rows, int32_t k_in, int32_t k_out,
                                  int64_t *out_ids, float *out_u, int32_t *err_word,
                                  void *stream);

/*
 * Draft-to-target id remap.
 * vLLM Qwen3DSparkForCausalLM.map_draft_to_target: d2t holds offsets, so
 *   target_ids[i] = draft_ids[i] + d2t[draft_ids[i]];
 * with d2t == NULL the map is the identity.  A table exists exactly for a
 * pruned draft (draft_vocab < target_vocab, the `<` predicate of the same PR).
 *
 * draft_ids, target_ids  device int64 [n] (may alias: in-place is allowed).
 * d2t                    device int64 [draft_vocab] or NULL.
 * Errors: d2t == NULL while draft_vocab < target_vocab, or d2t != NULL while
 *         draft_vocab >= target_vocab -> INVALID_ARG.  An id outside
 *         [0, draft_vocab) or a result outside [0, target_vocab) writes 0 and
 *         sets DFLASH2_DEVERR_ID_RANGE.
 */
dflash2_status dflash2_d2t_remap(const int64_t *draft_ids, const int64_t *d2t, int64_t n,
                                 int64_t draft_vocab, int64_t target_vocab,
                                 int64_t *target_ids, int32_t *err_word, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H */
