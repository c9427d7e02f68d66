/*
 * maxsim.h -- C ABI of the fused MaxSim library for GB300 (sm_103a).
 *
 * The operator (late interaction, ColBERT / ColPali):
 *
 *     score[i, j] = sum_s  max_t  < Q[i, s], D[j, t] >
 *
 * ("Flash-MaxSim" paper, Sec. 1, Eq. (1); "late-interaction-kernels" design
 * notes, section "Problem"). The [Lq, Ld] similarity tile of a pair lives only
 * in tensor memory and registers; it is never written to device memory.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller. Tensors are
 *    contiguous and row-major with the embedding dimension innermost. Q, D,
 *    scale and gradient (dQ, dD) pointers must be 16-byte aligned; row
 *    strides are dim elements.
 *  - Masks are one byte per token, nonzero = active. A masked document token
 *    is set to -inf before the max; a masked query token contributes 0 to the
 *    sum (design notes, "Problem" and "Mask handling").
 *  - argmax uses the lowest index among equal maxima (design notes,
 *    "Backward"). A query row with no valid document token (an empty or fully
 *    masked document) contributes 0 and reports argmax -1.
 *  - Outputs are fully overwritten; callers need not clear them.
 *  - `workspace` is caller-owned device scratch of at least the size reported
 *    by maxsim_workspace_size() for the same shape (NULL is allowed when that
 *    size is 0). The library itself never allocates device memory.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    asynchronous; arguments are validated on the host before any launch and
 *    an invalid call returns an error without launching anything.
 *  - Device-side checks (a bounded wait that gave up, an out-of-range argmax
 *    handed to the backward, inconsistent cu_seqlens) never trap: the kernel
 *    records a code that maxsim_device_status() returns.
 *  - Sizes are int64; supported: dim a multiple of 16 in [16, 256] for
 *    f16 / bf16 (a multiple of 32 in [32, 256] for int8); every token count
 *    below 2^31.
 */
#ifndef MAXSIM_H
#define MAXSIM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MAXSIM_OK = 0,
    MAXSIM_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, negative size, bad dtype */
    MAXSIM_ERR_UNSUPPORTED = 2,  /* valid but outside the supported envelope (e.g. dim) */
    MAXSIM_ERR_CUDA = 3,         /* a CUDA runtime / driver call failed */
    MAXSIM_ERR_TIMEOUT = 4,      /* device: a bounded wait expired; results are invalid */
    MAXSIM_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
    MAXSIM_ERR_DEVICE_INPUT = 6  /* device: an input failed a device-side check */
} maxsim_status;

typedef enum { MAXSIM_F16 = 0, MAXSIM_BF16 = 1 } maxsim_dtype;

/* Operation codes for maxsim_workspace_size(). */
enum { MAXSIM_OP_FWD = 0, MAXSIM_OP_FWD_VARLEN = 1, MAXSIM_OP_BWD = 2, MAXSIM_OP_FWD_INT8 = 3,
       MAXSIM_OP_SCORE_PAIRS = 4, MAXSIM_OP_CHAMFER_FWD = 5, MAXSIM_OP_CHAMFER_BWD = 6,
       MAXSIM_OP_TWO_STAGE = 7, MAXSIM_OP_FWD_STREAMED = 8, MAXSIM_OP_BWD_VARLEN = 9,
       MAXSIM_OP_FWD_VARLEN_STREAMED = 10 };

/*
 * Dense forward.
 *   Q       [Nq, Lq, dim]  f16 / bf16
 *   D       [Nd, Ld, dim]  same dtype
 *   q_mask  [Nq, Lq] u8 or NULL      d_mask [Nd, Ld] u8 or NULL
 *   scores  [Nq, Nd] f32 (out)
 *   argmax  [Nq * Nd, Lq] i32 (out, optional): row i*Nd + j, column s holds
 *           the winning document token t of query token s (0 <= t < Ld), or -1.
 * Computed with fp32 accumulation on the tensor cores ("late-interaction-
 * kernels" design notes, "Forward" and "Numerical accuracy"). Queries longer
 * than 512 tokens are split into chunks whose partial scores are summed
 * (notes, "Long-query chunking"); dim > 128 accumulates the partial dot
 * products of successive 128-wide slices before the max.
 */
maxsim_status maxsim_fwd(const void *Q, const void *D, maxsim_dtype dtype,
                         int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim,
                         const uint8_t *q_mask, const uint8_t *d_mask,
                         float *scores, int32_t *argmax,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * Padding-free forward over packed documents ("Flash-MaxSim" Sec. 4.3.2;
 * design notes, "Varlen / packed path").
 *   Q             dense [Nq, max_lq, dim] when cu_seqlens_q is NULL, else
 *                 packed [cu_seqlens_q[Nq], dim]
 *   cu_seqlens_q  [Nq + 1] i32 or NULL (FlashAttention convention: query i
 *                 owns rows cu[i] .. cu[i+1]-1, cu[0] = 0, non-decreasing)
 *   D             packed [total_d, dim]; document j owns rows
 *                 cu_seqlens_d[j] .. cu_seqlens_d[j+1]-1
 *   cu_seqlens_d  [Nd + 1] i32, cu[0] = 0, cu[Nd] = total_d
 *   max_lq        the longest query (upper bound on every query length)
 *   q_mask        one byte per query row of Q's layout, or NULL
 *   d_mask        [total_d] u8 or NULL
 *   scores        [Nq, Nd] f32 (out); an empty document scores 0
 *   argmax        [Nq * Nd, max_lq] i32 (out, optional); t is relative to the
 *                 document's first row; -1 beyond the query's length.
 * Work is proportional to the real tokens (sum of lengths), not Nd * max_ld.
 * cu_seqlens are checked on the device (MAXSIM_ERR_DEVICE_INPUT).
 */
maxsim_status maxsim_fwd_varlen(const void *Q, const int32_t *cu_seqlens_q, int64_t max_lq,
                                const void *D, const int32_t *cu_seqlens_d, int64_t total_d,
                                maxsim_dtype dtype, int64_t Nq, int64_t Nd, int64_t dim,
                                const uint8_t *q_mask, const uint8_t *d_mask,
                                float *scores, int32_t *argmax,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * Forward for an arbitrary list of (query, document) pairs of the packed
 * batches of maxsim_fwd_varlen, output [num_pairs] instead of [Nq, Nd]
 * (design notes, "Varlen / packed path": score_pairs_packed; for pair lists
 * sparse relative to Nq x Nd, as in reranker scheduling).
 *   Q, cu_seqlens_q, max_lq, D, cu_seqlens_d, total_d, dtype, Nq, Nd, dim,
 *   q_mask, d_mask   as for maxsim_fwd_varlen
 *   pairs      [num_pairs, 2] i32, pairs[p] = (query index, document index)
 *   scores     [num_pairs] f32 (out): the score of pair p
 *   argmax     [num_pairs, max_lq] i32 (out, optional), layout as a row of
 *              maxsim_fwd_varlen's argmax
 * The pairs are grouped by query on the device; every pair streams its own
 * document, so a document named by several pairs is read once per pair.
 * Results per pair equal maxsim_fwd_varlen's entry (i, j). A pair with an
 * index outside [0, Nq) x [0, Nd) scores 0 (argmax row -1) and is reported as
 * MAXSIM_ERR_DEVICE_INPUT by maxsim_device_status(). Queries up to 512 tokens
 * (at dim <= 128; MAXSIM_ERR_UNSUPPORTED beyond). Workspace:
 * maxsim_workspace_size(MAXSIM_OP_SCORE_PAIRS, Nq, max_lq, Nd, num_pairs, dim).
 */
maxsim_status maxsim_score_pairs_packed(const void *Q, const int32_t *cu_seqlens_q, int64_t max_lq,
                                        const void *D, const int32_t *cu_seqlens_d, int64_t total_d,
                                        maxsim_dtype dtype, int64_t Nq, int64_t Nd, int64_t dim,
                                        const uint8_t *q_mask, const uint8_t *d_mask,
                                        const int32_t *pairs, int64_t num_pairs,
                                        float *scores, int32_t *argmax,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward through the saved argmax ("Flash-MaxSim" Sec. 4.2, Eqs. (2)-(3);
 * design notes, "Backward"), for dense Q / D:
 *   dQ[i,s] = q_mask[i,s] * sum_j g[i,j] * D[j, argmax[i*Nd+j, s]]
 *   dD[j,t] = sum over (i,s) with argmax[i*Nd+j, s] == t of q_mask[i,s]*g[i,j]*Q[i,s]
 *   argmax       [Nq * Nd, Lq] i32 from maxsim_fwd (values in [-1, Ld))
 *   grad_scores  [Nq, Nd] f32
 *   dQ           [Nq, Lq, dim] f32 (out, optional)
 *   dD           [Nd, Ld, dim] f32 (out, optional)
 *   csr_row_ptr  [Nd * Ld + 1] i32 (out, optional): exclusive prefix sum of the
 *                number of sources that selected each document token
 *   csr_col      [Nq * Nd * Lq] i32 (out, optional): for each destination, its
 *                sources p = (i*Nd + j)*Lq + s in ascending order (first
 *                csr_row_ptr[Nd*Ld] entries written)
 * dD is reduced destination by destination from the inverse-argmax CSR with
 * no atomics (Sec. 4.2.2-4.2.3); dQ is reduced row by row in ascending j.
 * Both are bitwise reproducible. Sources with argmax -1 contribute nothing;
 * an argmax outside [-1, Ld) is skipped and reported as
 * MAXSIM_ERR_DEVICE_INPUT by maxsim_device_status(). When both dQ and dD (or
 * the CSR) are asked for, dQ runs on a stream the library owns beside
 * `stream`, forked after the work already on `stream` and joined back before
 * the call returns: work enqueued on `stream` afterwards sees both results.
 */
maxsim_status maxsim_bwd(const void *Q, const void *D, maxsim_dtype dtype,
                         int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim,
                         const uint8_t *q_mask, const int32_t *argmax, const float *grad_scores,
                         float *dQ, float *dD, int32_t *csr_row_ptr, int32_t *csr_col,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * INT8 x INT8 forward with per-token symmetric scales ("Flash-MaxSim"
 * Sec. 4.3.1: dequantisation fused into the kernel):
 *   dot[s,t] = sum_k Q8[i,s,k] * D8[j,t,k]   (exact integer)
 *   m_s      = max_t dot[s,t] * d_scale[j,t] (valid t only)
 *   score    = sum_s q_mask * q_scale[i,s] * m_s
 *   Q [Nq, Lq, dim] i8, q_scale [Nq, Lq] f32 (> 0)
 *   D [Nd, Ld, dim] i8, d_scale [Nd, Ld] f32 (> 0)
 *   argmax  [Nq * Nd, Lq] i32 (out, optional)
 *   win_dot [Nq * Nd, Lq] i32 (out, optional; needs argmax): the exact dot at
 *   the argmax (0 where argmax is -1).
 * The tensor cores of sm_103a have no 8-bit integer MMA kind: the INT8 tiles
 * are converted to binary16 in shared memory (exact for |v| <= 127) and
 * accumulated in fp32, which is exact for |dot| < 2^24.
 * The integer products are exact (|dot| < 2^24 for dim <= 256 with values in
 * [-127, 127]).
 */
maxsim_status maxsim_fwd_int8(const int8_t *Q, const float *q_scale,
                              const int8_t *D, const float *d_scale,
                              int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim,
                              const uint8_t *q_mask, const uint8_t *d_mask,
                              float *scores, int32_t *argmax, int32_t *win_dot,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Chamfer distance ("Flash-MaxSim" paper, Sec. 4.2.4, the generalisation of
 * the hard-selection pattern to a min over squared Euclidean distances) of B
 * independent pairs of point sets:
 *   CD(P_b, Q_b) = (1/N) sum_p min_q ||p - q||^2 + (1/M) sum_q min_p ||q - p||^2
 *   P       [B, N, dim] f32        Q [B, M, dim] f32        1 <= dim <= 8
 *   dist_p  [B, N] f32 (out): squared distance from each p to its nearest q
 *   idx_p   [B, N] i32 (out): the index in [0, M) of that q
 *   dist_q, idx_q [B, M] (out): the same from Q to P
 *   loss    [B] f32 (out): CD(P_b, Q_b)
 * The [N, M] distance table is never formed (online min over streamed
 * tiles). The nearest point is searched in fp32 on ||y||^2 - 2 <x, y>; among
 * candidates whose fp32 values are equal the lowest index wins; dist is then
 * computed directly as sum_k (x_k - y_k)^2 in fp32 and the loss sums it in
 * double. With an empty set (N or M = 0) the loss is 0 and every point of the
 * other set reports index -1 and distance 0. Coordinates must be finite and
 * their squared norms representable in fp32. P, Q and the outputs need 4-byte
 * alignment, the workspace 256-byte alignment. Workspace:
 * maxsim_workspace_size(MAXSIM_OP_CHAMFER_FWD, B, N, M, 0, dim).
 */
maxsim_status maxsim_chamfer_fwd(const float *P, const float *Q, int64_t B, int64_t N, int64_t M, int64_t dim,
                                 float *dist_p, int32_t *idx_p, float *dist_q, int32_t *idx_q, float *loss,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Gradient of sum_b grad_loss[b] * CD(P_b, Q_b) through the saved nearest
 * indices a = idx_p, c = idx_q of maxsim_chamfer_fwd (Sec. 4.2.4 with the
 * inverse index of Sec. 4.2.2 and the destination-owned reduction of 4.2.3):
 *   dP[p] = g (2/N) (p - Q[a_p]) - g (2/M) sum over q with c_q = p of (q - p)
 *   dQ[q] = g (2/M) (q - P[c_q]) - g (2/N) sum over p with a_p = q of (p - q)
 *   idx_p [B, N] i32, idx_q [B, M] i32 (values in [-1, size of the other set))
 *   grad_loss [B] f32;  dP [B, N, dim] f32 (out);  dQ [B, M, dim] f32 (out)
 * The inverse maps are built on the device as a CSR by a stable sort of the
 * flattened destinations; every gradient row is written by one thread that
 * sums its inverse row in ascending source order: no atomics, bitwise
 * reproducible. fp32 arithmetic. An index of -1 contributes nothing; an index
 * outside [-1, size) is skipped and reported as MAXSIM_ERR_DEVICE_INPUT by
 * maxsim_device_status(). Workspace:
 * maxsim_workspace_size(MAXSIM_OP_CHAMFER_BWD, B, N, M, 0, dim).
 */
maxsim_status maxsim_chamfer_bwd(const float *P, const float *Q, int64_t B, int64_t N, int64_t M, int64_t dim,
                                 const int32_t *idx_p, const int32_t *idx_q, const float *grad_loss, float *dP,
                                 float *dQ, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Top-k of every row of a score matrix (the retrieval step after scoring:
 * TileMaxSim paper, "End-to-End Retrieval Latency"; the top-K scan among the
 * forward variants of "Flash-MaxSim" Sec. 4).
 *   scores      [rows, n] f32 (device)
 *   top_idx     [rows, k] i32 (out): column indices of the k largest values,
 *               by descending value, the lower index first among equal values
 *               (-0.0 equals +0.0; NaN ranks below every number)
 *   top_scores  [rows, k] f32 (out, optional): those values
 * 1 <= k <= min(n, 4096). One block per row: a radix select of the k-th value
 * (four 8-bit passes), an index-ordered compaction, a bitonic sort.
 */
maxsim_status maxsim_topk(const float *scores, int64_t rows, int64_t n, int64_t k, int32_t *top_idx,
                          float *top_scores, void *stream);

/*
 * Two-stage INT8 -> f16 / bf16 top-k ("Flash-MaxSim" Sec. 4: the two-stage
 * INT8 -> FP16 top-K scan among the forward variants):
 *   1. s8 = maxsim_fwd_int8 scores of every (query, document) pair;
 *   2. the k1 best documents of each query by s8 (maxsim_topk order);
 *   3. those Nq * k1 pairs rescored from the f16 / bf16 embeddings
 *      (maxsim_score_pairs_packed on the dense corpus);
 *   4. the k best of each query's rescored candidates.
 *   Q8 [Nq, Lq, dim] i8 + q_scale [Nq, Lq] f32;  D8 [Nd, Ld, dim] i8 + d_scale [Nd, Ld] f32
 *   Q16 [Nq, Lq, dim], D16 [Nd, Ld, dim] in `dtype`: the same embeddings at 16 bits
 *   top_idx [Nq, k] i32 (out): document indices;  top_scores [Nq, k] f32 (out, optional)
 *   stage1_scores [Nq, Nd] f32 (out, optional): s8;  candidates [Nq, k1] i32 (out, optional)
 * dim a multiple of 32 up to 128 and Lq <= 512 (the rescoring stage holds one
 * query per unit); 1 <= k <= k1 <= min(Nd, 4096). No masks. Workspace:
 * maxsim_workspace_size(MAXSIM_OP_TWO_STAGE, Nq, Lq, Nd, Ld, dim), 256-byte aligned.
 */
maxsim_status maxsim_two_stage_topk(const int8_t *Q8, const float *q_scale, const int8_t *D8, const float *d_scale,
                                    const void *Q16, const void *D16, maxsim_dtype dtype, int64_t Nq, int64_t Lq,
                                    int64_t Nd, int64_t Ld, int64_t dim, int64_t k1, int64_t k, int32_t *top_idx,
                                    float *top_scores, float *stage1_scores, int32_t *candidates, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * Out-of-core dense forward ("Flash-MaxSim" Sec. 5.3): the corpus stays in
 * host memory and is scored in blocks of `block_docs` documents, so device
 * memory holds two blocks whatever the corpus size.
 *   Q       [Nq, Lq, dim] f16 / bf16, DEVICE pointer;  q_mask [Nq, Lq] u8 device or NULL
 *   D_host  [Nd, Ld, dim] same dtype, HOST pointer (page-locked memory lets the
 *           copies overlap the scoring; pageable memory is correct but slower)
 *   scores  [Nq, Nd] f32, device (out): equal to maxsim_fwd's
 * The copy of block b + 1 (cudaMemcpyAsync on a copy stream the library owns,
 * one per device) overlaps the forward of block b on `stream`; events order
 * the two. The call only enqueues: later work on `stream` sees the scores.
 * D_host must stay valid and unchanged until `stream` reaches that point.
 * Calls from several host threads are serialised inside the library. No
 * d_mask and no argmax. Workspace (two blocks, the block's scores, the
 * forward's own scratch; 256-byte aligned):
 * maxsim_workspace_size(MAXSIM_OP_FWD_STREAMED, Nq, Lq, block_docs, Ld, dim).
 */
maxsim_status maxsim_fwd_streamed(const void *Q, const void *D_host, maxsim_dtype dtype, int64_t Nq, int64_t Lq,
                                  int64_t Nd, int64_t Ld, int64_t dim, int64_t block_docs, const uint8_t *q_mask,
                                  float *scores, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward over packed layouts: the gradient of maxsim_fwd_varlen through its
 * saved argmax ("Flash-MaxSim" Sec. 4.2, Eqs. (2)-(3), on the packed layout of
 * Sec. 4.3.2; the pages' own varlen backward scatters with atomics, this one
 * keeps the destination-owned CSR reduction of Sec. 4.2.3).
 *   Q, cu_seqlens_q, max_lq   as for maxsim_fwd_varlen (dense Q when cu_seqlens_q is NULL)
 *   D [total_d, dim], cu_seqlens_d [Nd + 1]; max_ld >= every document length
 *   argmax       [Nq * Nd, max_lq] i32 from maxsim_fwd_varlen (t relative to the
 *                document's first row, -1 past a query's end)
 *   grad_scores  [Nq, Nd] f32;  q_mask one byte per query row of Q's layout, or NULL
 *   dQ           Q's layout, f32 (out, optional): packed [cu_seqlens_q[Nq], dim] or
 *                dense [Nq, max_lq, dim]
 *   dD           [total_d, dim] f32 (out, optional)
 *   csr_row_ptr  [total_d + 1] i32 (out, optional): CSR rows are D's packed rows
 *   csr_col      [Nq * Nd * max_lq] i32 (out, optional): sources p = (i*Nd + j)*max_lq + s
 * Deterministic, no atomics on the gradients. Inconsistent offsets, a document
 * longer than max_ld, or an argmax outside its document or past its query's end
 * are skipped and reported as MAXSIM_ERR_DEVICE_INPUT. As for maxsim_bwd, dQ
 * runs on a library-owned stream beside `stream` when dD or the CSR is also
 * asked for, joined back before the call returns. Workspace:
 * maxsim_workspace_size(MAXSIM_OP_BWD_VARLEN, Nq, max_lq, Nd, total_d, dim).
 */
maxsim_status maxsim_bwd_varlen(const void *Q, const int32_t *cu_seqlens_q, int64_t max_lq, const void *D,
                                const int32_t *cu_seqlens_d, int64_t total_d, int64_t max_ld, maxsim_dtype dtype,
                                int64_t Nq, int64_t Nd, int64_t dim, const uint8_t *q_mask, const int32_t *argmax,
                                const float *grad_scores, float *dQ, float *dD, int32_t *csr_row_ptr,
                                int32_t *csr_col, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Out-of-core packed forward ("Flash-MaxSim" Sec. 5.3 applied to the packed
 * layout of Sec. 4.3.2): maxsim_fwd_varlen over a corpus held in host memory.
 *   Q, cu_seqlens_q, max_lq, q_mask   DEVICE, as for maxsim_fwd_varlen
 *   D_host             packed [total_d, dim] rows, HOST memory (page-locked for overlap)
 *   cu_seqlens_d_host  [Nd + 1] i32, HOST memory; read by this call on the host
 *   block_docs, block_tokens   a block is the longest run of whole documents within
 *                      both limits; every document must fit block_tokens
 *   scores             [Nq, Nd] f32, device (out): equal to maxsim_fwd_varlen's
 * Block b + 1 is copied (rows and offsets, cudaMemcpyAsync on the library's
 * copy stream) while block b is scored on `stream`; the call only enqueues,
 * and the host buffers must stay valid until `stream` passes it. No d_mask
 * and no argmax. Workspace: maxsim_workspace_size(MAXSIM_OP_FWD_VARLEN_STREAMED,
 * Nq, max_lq, block_docs, block_tokens, dim), 256-byte aligned.
 */
maxsim_status maxsim_fwd_varlen_streamed(const void *Q, const int32_t *cu_seqlens_q, int64_t max_lq,
                                         const void *D_host, const int32_t *cu_seqlens_d_host, int64_t total_d,
                                         maxsim_dtype dtype, int64_t Nq, int64_t Nd, int64_t dim,
                                         const uint8_t *q_mask, int64_t block_docs, int64_t block_tokens,
                                         float *scores, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace an operation needs for a shape (0 if none).
 *   MAXSIM_OP_FWD / MAXSIM_OP_FWD_INT8: (Nq, Lq, Nd, Ld, dim)
 *   MAXSIM_OP_FWD_VARLEN:              (Nq, max_lq, Nd, total_d, dim); assumes
 *                                      packed Q (an upper bound for dense Q)
 *   MAXSIM_OP_BWD:                     (Nq, Lq, Nd, Ld, dim); assumes the CSR
 *                                      outputs are NULL (an upper bound)
 *   MAXSIM_OP_SCORE_PAIRS:             (Nq, max_lq, Nd, num_pairs, dim)
 *   MAXSIM_OP_CHAMFER_FWD / _BWD:      (B, N, M, 0, dim)
 *   MAXSIM_OP_TWO_STAGE:               (Nq, Lq, Nd, Ld, dim); enough for any
 *                                      k1 <= min(Nd, 4096)
 *   MAXSIM_OP_FWD_STREAMED:            (Nq, Lq, block_docs, Ld, dim); independent
 *                                      of the corpus size
 *   MAXSIM_OP_BWD_VARLEN:              (Nq, max_lq, Nd, total_d, dim); assumes
 *                                      the CSR outputs are NULL (an upper bound)
 *   MAXSIM_OP_FWD_VARLEN_STREAMED:     (Nq, max_lq, block_docs, block_tokens, dim);
 *                                      independent of the corpus size
 * Returns (size_t)-1 for an invalid shape.
 */
size_t maxsim_workspace_size(int op, int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim);

/* Static English description of a status code. */
const char *maxsim_status_string(maxsim_status status);

/*
 * Synchronises `stream`, then returns and clears the device-side status word
 * of the current device (MAXSIM_OK if no kernel recorded a problem).
 */
maxsim_status maxsim_device_status(void *stream);

/* The same call under the name the problem statement of this library uses. */
maxsim_status maxsim_last_device_status(void *stream);

/*
 * Fault-handling test hook (the papers have no counterpart): lets a test
 * drive a device-side bounded wait past its limit without faulting the GPU.
 * It arms a one-shot for the next forward-kernel launch from this process
 * (maxsim_fwd, _fwd_varlen, _fwd_int8, _score_pairs_packed and the calls
 * built on them): that launch's epilogue warps first wait on an mbarrier
 * that nothing ever arrives at and give up after limit_ns
 * (1 <= limit_ns <= 2e9, else MAXSIM_ERR_INVALID_ARG). Giving up records
 * MAXSIM_ERR_TIMEOUT in the device status word and raises the CTA's abort
 * flag; every other role stops at its next wait, the copies and MMAs already
 * issued are drained (each drain bounded by the normal 2 s limit), tensor
 * memory is freed and the kernel returns. The call itself returns MAXSIM_OK
 * and its outputs are invalid; the next call runs normally. Nothing traps
 * and no wait is endless.
 */
maxsim_status maxsim_debug_inject_wait_timeout(uint64_t limit_ns);

/*
 * Allocation-free variant of maxsim_fwd_varlen (the pages have no counterpart:
 * this is a deployment convenience of this library).
 *
 * Some callers cannot allocate device memory: a plugin inside a serving stack
 * that is handed only its input and output buffers, a C host with no device
 * allocator of its own or with a fixed memory budget that forbids a
 * cudaMalloc in the serving loop. They cannot provide the workspace that
 * maxsim_fwd_varlen needs for its repacked query rows. This entry point takes
 * the same arguments minus the workspace, and uses instead a scratch array of
 * MAXSIM_NOALLOC_SCRATCH_BYTES compiled into the library's device image. It
 * calls no cudaMalloc, cudaFree or allocating library routine.
 *  - The scratch exists on every GPU that loads the library, until exit.
 *  - The first call on a device looks up the array's device address (with that
 *    device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array, so calls that overlap on the
 *    GPU (other streams, other host threads) race on it: serialise them.
 *  - Shapes whose workspace (maxsim_workspace_size(MAXSIM_OP_FWD_VARLEN, ...))
 *    exceeds MAXSIM_NOALLOC_SCRATCH_BYTES return MAXSIM_ERR_UNSUPPORTED
 *    without launching; at dim = 128 that is about 64K padded query rows.
 * Results are identical to maxsim_fwd_varlen's for the same inputs.
 */
#define MAXSIM_NOALLOC_SCRATCH_BYTES (16u << 20)
maxsim_status maxsim_fwd_varlen_noalloc(const void *Q, const int32_t *cu_seqlens_q, int64_t max_lq,
                                        const void *D, const int32_t *cu_seqlens_d, int64_t total_d,
                                        maxsim_dtype dtype, int64_t Nq, int64_t Nd, int64_t dim,
                                        const uint8_t *q_mask, const uint8_t *d_mask,
                                        float *scores, int32_t *argmax, void *stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int maxsim_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAXSIM_H */
