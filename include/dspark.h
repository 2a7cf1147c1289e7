/*
 * dspark.h -- C ABI of the DSpark per-step speculative-decoding hot path on one
 * GB300 GPU (sm_103a).
 *
 * The method is described in "DSpark: Confidence-Scheduled Speculative
 * Decoding with Semi-Autoregressive Generation" (arXiv 2607.05147) and in the
 * tutorial "Speculative decoding, from zero to DSpark".  Section references
 * below are to those pages.
 *
 * Conventions for every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *     never allocates or frees device memory; scratch space is passed in as a
 *     caller-owned workspace whose size is given by the matching *_workspace_bytes
 *     query.  Tensors are dense, row-major, with the layouts stated per argument.
 *   - `stream` is a cudaStream_t passed as void*.  All work is enqueued
 *     asynchronously on that stream; the host never synchronises, except in
 *     dspark_check().
 *   - The return value reports HOST-side validation of sizes, pointers and
 *     dtypes, done before anything is launched.  On a non-zero return nothing was
 *     enqueued.
 *   - Errors that depend on device data (a token id out of range, lengths out of
 *     range, an inconsistent offset table, a too-short SPS table, a temperature
 *     out of range) are written to the caller's int32 `dev_status` word (the
 *     first error wins).  While *dev_status is non-zero every kernel of the
 *     library returns without doing work, so a failed step leaves its outputs
 *     unspecified and skips the rest.  dspark_check() synchronises the stream,
 *     returns the device status and resets the word to zero.
 *   - Logits and transition factors of one call share one dtype (DSPARK_F32 or
 *     DSPARK_BF16, dims.dtype).  Token ids are int32 in [0, V).
 *   - All randomness comes from one counter-based stream, Philox4x32-10
 *     (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11):
 *       key = (seed low 32 bits, seed high 32 bits),
 *       counter = (i >> 2, position, request, tag), word (i & 3) for stream index i,
 *       tag 0 = draft block noise (position k), 1 = accept uniform (position j,
 *       i = 0), 2 = residual / bonus block noise (the rejecting position j, or
 *       ell_r + 1 for the bonus), 3 and 4 = the in-block draws of tags 0 and 2;
 *       Gumbel uniform u = ((w >> 9) + 0.5) * 2^-23, g = -log(-log u);
 *       accept uniform u = (w >> 8) * 2^-24.
 *     Requests are identified by their index r in the call.
 *   - Categorical draws ("sample v with probability w_v / sum w"; the pages fix
 *     no mechanism) use a two-level draw over blocks of 32 indices: block
 *     g = v >> 5 with mass L_g enters a Gumbel race with score
 *     log L_g - log(-log u_g), u_g the Gumbel uniform of stream index g; the
 *     block with the largest score wins (ties to the smaller g), and inside it
 *     the first v whose running weight sum exceeds u'_g L_g is drawn, u'_g the
 *     accept uniform of stream index g of the in-block tag.  The draw has law
 *     w / sum(w) exactly and needs one random word per 32 indices.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_NULL = 1,            /* a required pointer is NULL                          */
  DSPARK_ERR_DIMS = 2,            /* B < 1, K_max not in 1..16, V < 2, rank < 1, sizes   */
  DSPARK_ERR_DTYPE = 3,           /* dtype not DSPARK_F32 / DSPARK_BF16                  */
  DSPARK_ERR_TEMPERATURE = 4,     /* device: temperature NaN, inf, < 0 or in (0, 1e-3)   */
  DSPARK_ERR_SPS_TOO_SHORT = 5,   /* device: sps_len < B + #candidates + 1               */
  DSPARK_ERR_OFFSETS = 6,         /* device: tgt_off[0] != 0 or a gap != ell_r + 1        */
  DSPARK_ERR_TOKEN_RANGE = 7,     /* device: an anchor / draft token outside [0, V)      */
  DSPARK_ERR_LENGTHS = 8,         /* device: K_r not in 1..K_max or ell_r not in 0..K_max */
  DSPARK_ERR_CONFIDENCE = 9,      /* device: a confidence outside [0, 1] or NaN          */
  DSPARK_ERR_WORKSPACE = 10,      /* workspace NULL, too small or not 256-byte aligned   */
  DSPARK_ERR_DEVICE_TIMEOUT = 11, /* device: a bounded wait inside a kernel gave up      */
  DSPARK_ERR_CUDA = 12,           /* a CUDA runtime call failed (launch, query, copy)    */
  DSPARK_ERR_UNSUPPORTED = 13,    /* the current device is not sm_103 / shape unsupported */
  DSPARK_ERR_BOUNDS = 14          /* device, bounds-checked build only: an index the kernels
                                     computed fell outside its buffer (the access was sent to
                                     element 0 instead); never returned by the normal build */
} dspark_status;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

/* dims.flags bits */
#define DSPARK_FLAG_FORCE_SIMT 1u /* draft: use the CUDA-core bias path even when the tensor-core path applies */
#define DSPARK_FLAG_W_PACKED 2u   /* draft: W is the packed projection of dspark_draft_pack_projection */
#define DSPARK_FLAG_SPARE_SM 4u   /* draft: the tensor-core path leaves one SM free, so that a kernel on
                                     another stream (the scheduler) runs beside it */
#define DSPARK_FLAG_TEST_BARRIER_TIMEOUT 8u /* draft, tensor-core path, for testing the failure path only:
                                     the grid barrier before position 2 waits for one arrival more than
                                     the grid gives, so the bounded wait runs out (about 2 s), the kernel
                                     drains what it issued, frees its tensor memory and the call reports
                                     DSPARK_ERR_DEVICE_TIMEOUT through the device status word */

typedef struct {
  int64_t B;      /* requests in the call                                  */
  int64_t K_max;  /* block size: draft positions per request, 1..16        */
  int64_t V;      /* vocabulary size                                       */
  int64_t rank;   /* Markov-head rank r (draft only; ignored by verify)     */
  int32_t dtype;  /* dspark_dtype of every logits / factor tensor           */
  uint32_t flags; /* DSPARK_FLAG_* bits                                    */
} dspark_dims;

/* ------------------------------------------------------------------------
 * Draft: Markov-head semi-autoregressive sampling ("DSpark" S3.1, Markov head;
 * "Speculative decoding, from zero to DSpark" S6).
 *
 * For each request r and position k = 1..K_r[r], left to right:
 *   z_k(v) = U[r, k-1, v] + sum_i E[x_{k-1}, i] * W[i, v]     (x_0 = anchor[r])
 *   stored in the call dtype (bf16 values are rounded to nearest even), then
 *   x_k ~ softmax(z_k / T_r) by the two-level draw (streams tag 0 and 3,
 *   position k)                                                (T_r > 0)
 *   x_k = argmax_v z_k(v), ties to the smallest v              (T_r = 0)
 *
 *   U            [B, K_max, V]  base logits of the parallel backbone.
 *   E            [V, rank]      W1, the Markov embedding table (row per previous token).
 *   W            [rank, V]      W2, the logit projection; or, with
 *                DSPARK_FLAG_W_PACKED, the packed projection written by
 *                dspark_draft_pack_projection (tensor-core path only).
 *   anchor       [B] int32      x_0, the previous round's bonus/correction token.
 *   K_r          [B] int32      draft length per request, 1..K_max.
 *   temperature  [B] float      T_r: 0 (greedy) or >= 1e-3.
 *   draft_tok    [B, K_max] int32 out: x_1..x_{K_r}; entries k > K_r are set to -1.
 *   draft_logits [B, K_max, V]  out, optional (NULL = not written): z_k, the logits
 *                actually sampled from; rows k > K_r are not written.
 *   draft_lse    [B, K_max] float out, optional: log sum_v exp(z_k(v) / T_r), the
 *                draft distribution's normaliser (for T_r = 0: max_v z_k(v));
 *                entries k > K_r are not written.
 *   draft_tok_logit [B, K_max] float out, optional: z_k(x_k), the stored-dtype logit
 *                of the drawn token (exact, as a float); entries k > K_r are not
 *                written.  With draft_lse it gives log q_k(x_k) = z_k(x_k) / T_r -
 *                lse, all that verification needs of a draft row except at a
 *                rejection, so draft_logits can stay NULL: no B x K x V logits go
 *                back to memory, and dspark_verify_markov recomputes the rejecting
 *                rows.
 *   workspace    >= dspark_draft_workspace_bytes(dims) bytes (the same dims and
 *                flags as the call), 256-byte aligned.
 * The tensor-core path is used when dtype = DSPARK_BF16, rank is a multiple of
 * 64 and <= 256, V is a multiple of 8, U, E, W and draft_logits are 16-byte
 * aligned and the device is sm_103; otherwise (or with DSPARK_FLAG_FORCE_SIMT)
 * the CUDA-core path runs.  Without DSPARK_FLAG_W_PACKED the tensor-core path
 * first packs W into the workspace (one read and one write of W per call);
 * weights that stay fixed across calls should be packed once instead.  A packed
 * W with a call that cannot take the tensor-core path returns
 * DSPARK_ERR_UNSUPPORTED.  Both paths give the same tokens except where a
 * decision is within fp32 rounding.
 * ------------------------------------------------------------------------ */
size_t dspark_draft_workspace_bytes(dspark_dims dims);

/* ------------------------------------------------------------------------
 * Packed projection for the tensor-core draft path (no counterpart on the
 * pages: a storage layout of W2 = W).
 *
 * W_packed holds rank/64 x ceil(V/64) blocks of 8 KB; block (c, t), at byte
 * offset (c * ceil(V/64) + t) * 8192, holds W[64c + i, 64t + n] for i, n < 64 as
 * 64 rows of 128 bytes (row i = rank index 64c + i), and within row i the 16-byte
 * unit at position u holds columns 64t + 8 (u ^ (i & 7)) .. + 7 (the 128-byte
 * swizzle of the tensor-core operand).  Columns past V are zero.
 *   dspark_draft_packed_projection_bytes: the size, or 0 when rank is not a
 *     multiple of 64 in 64..256 or V is not a multiple of 8.
 *   dspark_draft_pack_projection: W [rank, V] bf16 (dims.rank, dims.V, dims.dtype;
 *     16-byte aligned) -> W_packed (256-byte aligned, >= the size).  Errors:
 *     DSPARK_ERR_UNSUPPORTED for shapes or dtypes without a packed layout,
 *     DSPARK_ERR_WORKSPACE for a short or misaligned W_packed.
 * ------------------------------------------------------------------------ */
size_t dspark_draft_packed_projection_bytes(int64_t rank, int64_t V);

dspark_status dspark_draft_pack_projection(const void *W, dspark_dims dims, void *W_packed, size_t packed_bytes,
                                           void *stream);

dspark_status dspark_draft_markov_sample(const void *U, const void *E, const void *W,
                                         const int32_t *anchor, const int32_t *K_r,
                                         const float *temperature, uint64_t seed, dspark_dims dims,
                                         int32_t *draft_tok, void *draft_logits, float *draft_lse,
                                         float *draft_tok_logit, void *workspace, size_t workspace_bytes,
                                         int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Draft with the confidence head's Markov term fused in ("DSpark" S3.2.1;
 * "Speculative decoding, from zero to DSpark" S8).
 *
 * The confidence head is one linear projection of [h_k ; W1[x_{k-1}]] and a
 * sigmoid.  Its backbone part has no sequential dependence and is an input; its
 * Markov part needs the token sampled at position k-1, which this call has at
 * hand, so the head is evaluated inside the draft:
 *   conf[r, k] = sigmoid(conf_h[r, k] + sum_i conf_w[i] * E[x_{k-1}, i])
 * (x_0 = anchor[r]), fp32 arithmetic.  Every other argument, output and error is
 * that of dspark_draft_markov_sample, whose outputs are unchanged.
 *
 *   conf_h   [B, K_max] float  the backbone term w_h . h_k + b of the head.
 *   conf_w   [rank] float      the head's weights on the Markov embedding.
 *   conf     [B, K_max] float out: c_k for k <= K_r, 0 for k > K_r.
 * ------------------------------------------------------------------------ */
dspark_status dspark_draft_markov_sample_confidence(const void *U, const void *E, const void *W,
                                                    const int32_t *anchor, const int32_t *K_r,
                                                    const float *temperature, uint64_t seed, dspark_dims dims,
                                                    const float *conf_h, const float *conf_w,
                                                    int32_t *draft_tok, void *draft_logits, float *draft_lse,
                                                    float *draft_tok_logit, float *conf, void *workspace,
                                                    size_t workspace_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Draft with the RNN head ("DSpark" S3.1, RNN head).
 *
 * The Markov head's W1 row is replaced by the output of a gated recurrent cell
 * whose state s_k (size rank, s_0 = 0) carries the whole prefix of the block.
 * The paper's update equation is not printed; this library's reading: one
 * linear projection of [s_{k-1}; W1[x_{k-1}]; h_k], split into gate, candidate
 * and output parts,
 *   pre = rnn_x[r, k] + rnn_W [s_{k-1}; E[x_{k-1}]]       (3 rank values)
 *   g = sigmoid(pre[0:r]), c = tanh(pre[r:2r]), o = sigmoid(pre[2r:3r])
 *   s_k = g * s_{k-1} + (1 - g) * c,   f_k = o * s_k
 *   z_k(v) = U[r, k-1, v] + sum_i f_k[i] * W[i, v], then the draw as for the
 *   Markov head (same random streams), fp32 arithmetic.
 *
 *   rnn_W   [3 rank, 2 rank]   call dtype; rows: gate, candidate, output; columns
 *           0..rank-1 act on the state, rank..2 rank-1 on E[x_{k-1}].
 *   rnn_x   [B, K_max, 3 rank] float: the backbone term W_h h_k + b (no
 *           sequential dependence, computed with the backbone).
 *   workspace >= dspark_draft_rnn_workspace_bytes(dims), 256-byte aligned.
 * Every other argument is that of dspark_draft_markov_sample.  The call runs on
 * the CUDA-core path (W as given, rank <= 4096); DSPARK_FLAG_W_PACKED returns
 * DSPARK_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------ */
size_t dspark_draft_rnn_workspace_bytes(dspark_dims dims);

dspark_status dspark_draft_rnn_sample(const void *U, const void *E, const void *W, const void *rnn_W,
                                      const float *rnn_x, const int32_t *anchor, const int32_t *K_r,
                                      const float *temperature, uint64_t seed, dspark_dims dims,
                                      int32_t *draft_tok, void *draft_logits, float *draft_lse,
                                      float *draft_tok_logit, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Schedule: hardware-aware prefix scheduler ("DSpark" S3.2.2, Algorithm 1;
 * "Speculative decoding, from zero to DSpark" S8).
 *
 *   a[r, j] = prod_{i <= j} conf[r, i]     (sequential fp32 product, j = 1..K_r[r])
 *   candidates {(r, j) : a[r, j] > 0}, ranked by a descending, ties to the smaller
 *   position j, then the smaller request r;
 *   walking that order with B <- R + i and tau_i = R + sum of the first i values of
 *   a (exact 2^-40 fixed point), Theta_i = tau_i * SPS[R + i] (fp64, Theta_0 =
 *   R * SPS[R]); admit while Theta_i > Theta_{i-1}; stop at the first decline.
 *   ell[r] = number of admitted candidates of request r.
 *
 *   conf        [B, K_max] float  per-position acceptance confidences in [0, 1].
 *   K_r         [B] int32         draft lengths, 1..K_max.
 *   sps         [sps_len] double  SPS table indexed by verify batch tokens (entry 0
 *               unused); must hold every index up to B + #candidates.
 *   ell         [B] int32 out     scheduled verification lengths.
 *   tgt_off     [B+1] int32 out   exclusive scan of (ell + 1): row offsets of the
 *               flattened target logits consumed by dspark_verify_ragged.
 *   theta_best  [1] double out, optional: the objective at the stop.
 *   b_star      [1] int64 out, optional: the verify batch size R + sum(ell).
 *   survival    [B, K_max] float out, optional: a (0 for j > K_r).
 *   workspace   >= dspark_schedule_workspace_bytes(B, K_max) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------ */
size_t dspark_schedule_workspace_bytes(int64_t B, int64_t K_max);

dspark_status dspark_schedule_survival(const float *conf, const int32_t *K_r, const double *sps,
                                       int64_t sps_len, int64_t B, int64_t K_max, int32_t *ell,
                                       int32_t *tgt_off, double *theta_best, int64_t *b_star,
                                       float *survival, void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Deployed (asynchronous) scheduler, step 1: capacity ("DSpark" S5.2;
 * "Speculative decoding, from zero to DSpark" S9).
 *
 * Algorithm 1's ranking and objective with the early-stopping break removed:
 * Theta_i is evaluated for every i = 0..N along the greedy path (same survival
 * products, ranking, fixed-point tau and fp64 Theta as dspark_schedule_survival)
 * and the capacity is the i with the largest Theta_i, the smallest such i on
 * ties.  Called on the confidences of two steps earlier, it fixes how many draft
 * tokens the next verification pass admits, before that step's tokens exist, so
 * a global search across the SPS cliffs no longer leaks them.  The capacity
 * counts draft-token slots (the verify batch is B + capacity).
 *
 *   conf, K_r, sps, sps_len, B, K_max   as for dspark_schedule_survival.
 *   capacity    [1] int32 out          the admitted candidates at the maximum.
 *   theta_best  [1] double out, optional: Theta at the maximum.
 *   ell, tgt_off  out, optional (both or neither): the lengths of that admission
 *               (the retrospective schedule of Appendix A, for diagnostics).
 *   workspace   >= dspark_schedule_workspace_bytes(B, K_max) bytes, 256-byte aligned.
 * Errors as for dspark_schedule_survival.
 * ------------------------------------------------------------------------ */
dspark_status dspark_schedule_capacity(const float *conf, const int32_t *K_r, const double *sps,
                                       int64_t sps_len, int64_t B, int64_t K_max, int32_t *capacity,
                                       double *theta_best, int32_t *ell, int32_t *tgt_off, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Deployed (asynchronous) scheduler, step 2: dynamic top-K admission ("DSpark"
 * S5.2; "Speculative decoding, from zero to DSpark" S9).
 *
 * The current step's candidates are ranked exactly as in Algorithm 1 (survival
 * descending, ties to the smaller position, then the smaller request, so that a
 * token never moves its own rank) and the first min(*capacity, N) are admitted;
 * no SPS table is read.  ell[r] = admitted candidates of request r.
 *
 *   conf, K_r, B, K_max   as for dspark_schedule_survival.
 *   capacity    [1] int32, DEVICE: admitted draft tokens, >= 0 (for instance the
 *               output of dspark_schedule_capacity two steps earlier); a negative
 *               value is DSPARK_ERR_LENGTHS on the device.
 *   ell, tgt_off, b_star, survival   out as for dspark_schedule_survival
 *               (b_star, survival optional).
 *   workspace   >= dspark_schedule_workspace_bytes(B, K_max) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------ */
dspark_status dspark_schedule_topk(const float *conf, const int32_t *K_r, const int32_t *capacity, int64_t B,
                                   int64_t K_max, int32_t *ell, int32_t *tgt_off, int64_t *b_star,
                                   float *survival, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Static-threshold verification lengths: the baseline that "DSpark" S3.2.2
 * contrasts with its scheduler, and the threshold sweep of S4.3.3 (Fig. 5).
 *
 * ell[r] = the largest j <= K_r[r] such that every position i <= j passes:
 *   DSPARK_THRESHOLD_CONFIDENCE  conf[r, i] >= threshold,
 *   DSPARK_THRESHOLD_SURVIVAL    a[r, i] >= threshold (the survival products),
 * and a[r, i] > 0 (as in Algorithm 1's candidate pool).
 *
 *   conf, K_r, B, K_max   as for dspark_schedule_survival.
 *   threshold   any number but NaN (NaN: DSPARK_ERR_CONFIDENCE); <= 0 verifies
 *               every candidate, > 1 verifies nothing.
 *   mode        DSPARK_THRESHOLD_CONFIDENCE or DSPARK_THRESHOLD_SURVIVAL
 *               (otherwise DSPARK_ERR_DIMS).
 *   ell, tgt_off, b_star, survival   out as for dspark_schedule_survival
 *               (b_star, survival optional).
 * No workspace.
 * ------------------------------------------------------------------------ */
#define DSPARK_THRESHOLD_CONFIDENCE 0
#define DSPARK_THRESHOLD_SURVIVAL 1

dspark_status dspark_schedule_threshold(const float *conf, const int32_t *K_r, float threshold, int32_t mode,
                                        int64_t B, int64_t K_max, int32_t *ell, int32_t *tgt_off,
                                        int64_t *b_star, float *survival, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Schedule without a caller workspace.
 *
 * The paper has no counterpart to this entry point: it exists for callers that
 * cannot allocate device memory where they schedule -- a serving loop that must
 * not call cudaMalloc between steps (it synchronises the device), or a plugin
 * whose host process owns every device allocation and hands it no workspace.
 * It computes exactly what dspark_schedule_survival computes, with the same
 * arguments except the workspace, on scratch memory that is a static array of
 * this library (DSPARK_NOALLOC_SCRATCH_BYTES on every GPU that loads the
 * library, held until the process exits).  It allocates and frees nothing.
 *   - B * K_max must not exceed DSPARK_NOALLOC_MAX_CANDIDATES; larger calls
 *     return DSPARK_ERR_WORKSPACE and enqueue nothing.
 *   - The first call on a device (with that device current) looks up the
 *     scratch address once; make that first call before any stream capture.
 *   - Every call shares the one scratch array: calls whose kernels may overlap
 *     on the GPU (unordered streams) race on it.  Nothing in it needs clearing
 *     between calls.
 * ------------------------------------------------------------------------ */
#define DSPARK_NOALLOC_MAX_CANDIDATES 32768
#define DSPARK_NOALLOC_SCRATCH_BYTES (1088u * 1024u)

dspark_status dspark_schedule_survival_noalloc(const float *conf, const int32_t *K_r, const double *sps,
                                               int64_t sps_len, int64_t B, int64_t K_max, int32_t *ell,
                                               int32_t *tgt_off, double *theta_best, int64_t *b_star,
                                               float *survival, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Verify: ragged rejection-sampling verification ("DSpark" S2.1;
 * "Speculative decoding, from zero to DSpark" S2 and Appendix A1).
 *
 * For request r with temperature T and length ell_r, with
 *   q_j = softmax(draft_logits[r, j-1] / T),  p_j = softmax(tgt_logits[tgt_off[r]+j-1] / T):
 *   for j = 1..ell_r: accept x_j = draft_tok[r, j-1] iff u_j < min(1, p_j(x_j) / q_j(x_j)),
 *   u_j the accept uniform of (seed, j, r); stop at the first rejection and draw the
 *   correction from norm(max(0, p_j - q_j)) by the two-level draw on streams
 *   (seed, j, r, tags 2 and 4) (from p_j if no p_j(v) > q_j(v) in floating point); if
 *   every position is accepted, draw the bonus from softmax(z / T) of row
 *   tgt_off[r] + ell_r on streams (seed, ell_r + 1, r, tags 2 and 4).
 *   T = 0: accept iff x_j is the argmax of p_j; correction and bonus are argmaxes.
 *
 *   draft_logits [B, K_max, V]   the logits the drafts were sampled from.
 *   draft_lse    [B, K_max] float, optional: log-sum-exp of draft_logits / T per row
 *                (as written by dspark_draft_markov_sample).  When given, draft rows
 *                are read only at the rejecting position; when NULL they are
 *                streamed at every verified position.
 * The target rows are read position by position (every request's row j before any
 * row j + 1), and each row is decided as soon as its statistics are complete; rows
 * past a request's first rejection are skipped once that rejection is known (rows
 * already in flight are read anyway).
 *   tgt_logits   [tgt_off[B], V]  flattened target logits, ell_r + 1 rows per request.
 *   tgt_off      [B+1] int32      row offsets; tgt_off[r+1] - tgt_off[r] = ell_r + 1.
 *   ell          [B] int32        verification lengths, 0..K_max.
 *   draft_tok    [B, K_max] int32 draft tokens (entries j <= ell_r must lie in [0, V)).
 *   temperature  [B] float        as for the draft.
 *   n_acc        [B] int32 out    accepted draft tokens.
 *   out_tok      [B, K_max+1] int32 out: the n_acc accepted tokens, then the
 *                correction or bonus token, then -1.
 *   workspace    >= dspark_verify_workspace_bytes(B, V) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------ */
size_t dspark_verify_workspace_bytes(int64_t B, int64_t V);

dspark_status dspark_verify_ragged(const void *draft_logits, const float *draft_lse,
                                   const void *tgt_logits, const int32_t *tgt_off, const int32_t *ell,
                                   const int32_t *draft_tok, const float *temperature, uint64_t seed,
                                   dspark_dims dims, int32_t *n_acc, int32_t *out_tok,
                                   void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Verify with the draft rows recomputed ("DSpark" S2.1 and S3.1; "Speculative
 * decoding, from zero to DSpark" S2 and S6).
 *
 * The same verification as dspark_verify_ragged (same accept rule, random
 * streams and outputs) for drafts of the Markov head whose logits were not
 * stored: the accept test at position j needs only log q_j(x_j) =
 * draft_tok_logit / T - draft_lse, and the draft row of a rejecting position j
 * (T > 0) is recomputed for the residual as z = U[r, j-1] + E[x_{j-1}] . W,
 * rounded to bf16 exactly as the draft formed it (x_0 = anchor), by the
 * tensor-core path, so the residual is drawn from the very q that was sampled.
 * All rejections of a call share one pass over W.
 *
 *   U, E, W, anchor   as passed to dspark_draft_markov_sample (W as given, or
 *                     packed with DSPARK_FLAG_W_PACKED in dims.flags).
 *   draft_lse, draft_tok_logit  [B, K_max] float: the draft's outputs.
 *   tgt_logits, tgt_off, ell, draft_tok, temperature, seed, n_acc, out_tok
 *                     as for dspark_verify_ragged.
 *   dims              B, K_max, V and rank of the draft; dtype DSPARK_BF16.
 *   workspace         >= dspark_verify_markov_workspace_bytes(dims), 256-byte aligned.
 * Needs the tensor-core shape (bf16, rank a multiple of 64 up to 256, V a
 * multiple of 8, 16-byte aligned U, E, W and tgt_logits, an sm_103 device);
 * otherwise DSPARK_ERR_UNSUPPORTED (the workspace query returns 0), and
 * dspark_verify_ragged with stored draft logits serves the call.
 * ------------------------------------------------------------------------ */
size_t dspark_verify_markov_workspace_bytes(dspark_dims dims);

dspark_status dspark_verify_markov(const void *U, const void *E, const void *W, const int32_t *anchor,
                                   const float *draft_lse, const float *draft_tok_logit,
                                   const void *tgt_logits, const int32_t *tgt_off, const int32_t *ell,
                                   const int32_t *draft_tok, const float *temperature, uint64_t seed,
                                   dspark_dims dims, int32_t *n_acc, int32_t *out_tok, void *workspace,
                                   size_t workspace_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Status helpers.
 * ------------------------------------------------------------------------ */
/* Static, human-readable name of a status code ("DSPARK_OK", ...). */
const char *dspark_status_string(dspark_status s);

/* Synchronise `stream`, read *dev_status (a device int32), reset it to 0 and
 * return it.  Returns DSPARK_ERR_CUDA when the copy or the synchronisation fails. */
dspark_status dspark_check(int32_t *dev_status, void *stream);

/* ABI version of this header (major * 100 + minor): 200 added draft_tok_logit to the
 * draft entry points. */
int dspark_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
