/*
 * attnres.h -- C ABI of libattnres.so, the GB300 (sm_103a) implementation of
 * the Attention Residuals depth-wise softmax read.
 *
 * The operation (Full AttnRes; b-lab.team summary of "Attention Residuals",
 * section 1): for every token, a layer's input is
 *
 *     h = sum_i alpha_i v_i,   alpha_i = exp(w . RMSNorm(v_i)) / sum_j exp(w . RMSNorm(v_j)),
 *     RMSNorm(x) = g * x / sqrt(mean(x^2) + eps),
 *
 * over stored source rows v_i (the embedding, earlier layer or block
 * outputs), with a learned per-layer pseudo-query w.  The weighted sum uses
 * the raw source values; RMSNorm only enters the score.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every tensor pointer is a DEVICE pointer, row-major and
 *   contiguous, except that consecutive sources are src_stride elements
 *   apart.  Host pointers are named as such (only msar_expand_fwd's ksizes).
 *   The caller owns every buffer; the library allocates nothing, keeps no
 *   per-call state and is safe to call from several host threads.
 * Sources.  src holds n_src sources; source i is the [T, d] row block at
 *   src + i * src_stride (elements).  src_stride >= T * d.
 * Types.  dt selects the storage type of sources, partial sums and outputs:
 *   ATTNRES_F32 (float) or ATTNRES_BF16 (bfloat16).  Queries, gains and lse
 *   are always float.  All arithmetic is float32 (accumulation included);
 *   bf16 outputs are rounded to nearest-even once, at the store.
 * Gain.  gain is the RMSNorm gain g[d] (per head slice for MHAR) or NULL for
 *   all ones.  eps >= 0 is added to the mean square inside the square root.
 *   A zero key with eps = 0 normalises to zero (score 0).
 * Streams.  stream is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream).  Every call only enqueues work on it and returns.
 * Alignment and sizes.  d % 8 == 0; every tensor pointer 16-byte aligned
 *   (lse: 4-byte); src_stride * sizeof(element) a multiple of 16 bytes.
 * Errors.  Arguments are validated on the host before anything is launched;
 *   nothing aborts.  ATTNRES_ERR_INVALID_ARG: a NULL required pointer,
 *   T < 0, n_src < 1, d < 1, eps < 0 or NaN, src_stride < T*d, a head count
 *   that does not divide d, or an output that overlaps an input it must not
 *   alias.  ATTNRES_ERR_UNSUPPORTED: a valid request outside what the
 *   kernels implement (alignment, d % 8, n_q > 8, size limits listed per
 *   function).  ATTNRES_ERR_CUDA: a CUDA runtime call failed; the message is
 *   in attnres_last_cuda_error().  T == 0 is a no-op that returns ATTNRES_OK once
 *   the scalar arguments are valid; tensor pointers may then be NULL.
 *   ATTNRES_OK means the work was enqueued.  A device-side wait that ran out
 *   of time (ATTNRES_ERR_TIMEOUT) is reported by attnres_sync_status().
 */
#ifndef ATTNRES_H
#define ATTNRES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTNRES_F32 = 0, ATTNRES_BF16 = 1 } attnres_dtype_t;

typedef enum {
    ATTNRES_OK = 0,
    ATTNRES_ERR_INVALID_ARG = 1,
    ATTNRES_ERR_UNSUPPORTED = 2,
    ATTNRES_ERR_CUDA = 3,
    ATTNRES_ERR_TIMEOUT = 4
} attnres_status_t;

/*
 * Full AttnRes read of one layer.
 * Defined by: b-lab.team summary, section 1 (h_l = sum_{i<l} alpha_{i->l} v_i,
 * phi(q,k) = exp(q^T RMSNorm(k))); dimensionstp.github.io review, section
 * 3-2 1).  The layer's sources are v_0..v_{n_src-1}.
 *   src    [n_src][T][d] (stride src_stride), dtype dt
 *   query  [d] float, the layer's pseudo-query w_l
 *   gain   [d] float or NULL
 *   out    [T][d], dtype dt; must not overlap src
 * Any n_src >= 1 (sources beyond the on-chip chunk are folded in with an
 * online softmax).  Limits: d <= 16384 (bf16) / 8192 (f32).
 */
attnres_status_t attnres_full_fwd(const void *src, int64_t n_src, int64_t src_stride,
                                  int64_t T, int64_t d, attnres_dtype_t dt,
                                  const float *query, const float *gain, float eps,
                                  void *out, void *stream);

/*
 * Block AttnRes, phase 1 of the two-phase schedule: all n_q pseudo-queries of
 * a block read the n_src cached block representations in one pass, so each
 * cached b_n is read from memory once per block instead of once per layer.
 * Defined by: b-lab.team summary, section 3 (Inference, Phase 1: parallel
 * inter-block attention); dimensionstp.github.io review, section 3-2 4).
 * The softmax state of every (query, token) is returned normalised:
 *   o_q = sum_i e^{s_qi - m_q} v_i / l_q   and   lse_q = m_q + ln l_q,
 * so o_0 is already the input of the block's first layer (which reads no
 * partial sum: summary section 2, tutorial Fig. 4).
 *   src      [n_src][T][d] cached block representations b_0..b_{n-1}
 *   queries  [n_q][d] float, 1 <= n_q <= 8
 *   o        [n_q][T][d], dtype dt; must not overlap src
 *   lse      [n_q][T] float, or NULL if not needed
 * Limits: n_q * d <= 16384 after rounding n_q up to 1, 2, 4 or 8.
 */
attnres_status_t attnres_block_phase1(const void *src, int64_t n_src, int64_t src_stride,
                                      int64_t T, int64_t d, attnres_dtype_t dt,
                                      const float *queries, int64_t n_q,
                                      const float *gain, float eps,
                                      void *o, float *lse, void *stream);

/*
 * Block AttnRes, phase 2: fold one layer's intra-block partial-sum source into
 * its phase-1 state with the online-softmax merge (exact).
 * Defined by: b-lab.team summary, section 3 (Phase 2: sequential intra-block
 * attention + online softmax merge); dimensionstp.github.io review, 3-2 4).
 *   s_p = w . RMSNorm(p),  M = max(lse, s_p),
 *   out = (e^{lse-M} o + e^{s_p-M} p) / (e^{lse-M} + e^{s_p-M}).
 *   o        [T][d] dtype dt (one query's slice of phase-1 o)
 *   lse      [T] float (the matching slice of phase-1 lse)
 *   partial  [T][d] dtype dt, the block's current partial sum b^{(n)}_{i-1};
 *            NULL for the first layer of a block (then out = o)
 *   query    [d] float, the layer's pseudo-query
 *   out      [T][d] dtype dt; may be o itself (in place), must not overlap
 *            partial or partially overlap o
 */
attnres_status_t attnres_block_phase2_merge(const void *o, const float *lse,
                                            const void *partial, int64_t T, int64_t d,
                                            attnres_dtype_t dt, const float *query,
                                            const float *gain, float eps, void *out,
                                            void *stream);

/*
 * Block AttnRes, phase 2 fused with the intra-block partial-sum update: the
 * previous layer's output f joins the block's current partial sum, and the
 * next layer's merge scores the updated partial, in one pass (the partial is
 * read once instead of once by an update and again by the merge).
 * Defined by: b-lab.team summary, section 2 (the source of layer i >= 2 is
 * the partial sum b^{(n)}_{i-1} of the block's outputs so far) and section 3
 * (Phase 2, whose kernel fusion cuts I/O); ai-systems-engineering.com
 * tutorial, Fig. 4 (after a layer's output is produced only the current
 * partial sum changes, to the old partial plus that output).
 *   partial_out = partial + f       (partial NULL: partial_out = f),
 *   out = phase-2 merge of (o, lse) with partial_out, as
 *         attnres_block_phase2_merge.
 * The merge scores and mixes partial + f in fp32 (the exact sum of the two
 * stored inputs up to fp32 rounding); partial_out receives that sum rounded
 * once to dt, the value later layers and the next block read.
 *   partial      [T][d] dtype dt or NULL (the block's first output)
 *   f            [T][d] dtype dt, the previous layer's output
 *   partial_out  [T][d] dtype dt; may be partial or f itself, must not
 *                otherwise overlap them, o, out or lse
 *   o, lse       the next layer's phase-1 state ([T][d] dtype dt, [T] float)
 *   query        [d] float, the next layer's pseudo-query
 *   out          [T][d] dtype dt; may be o itself, must not overlap partial,
 *                f or partial_out
 */
attnres_status_t attnres_block_phase2_update_merge(const void *partial, const void *f,
                                                   void *partial_out, const void *o,
                                                   const float *lse, int64_t T, int64_t d,
                                                   attnres_dtype_t dt, const float *query,
                                                   const float *gain, float eps, void *out,
                                                   void *stream);

/*
 * MHAR, the multi-head block-diagonal read: the pseudo-query is reshaped into
 * H heads of d/H channels; each head has its own softmax over depth and mixes
 * only its own channel slice.  H = 1 is exactly attnres_block_phase1 (the same
 * kernel runs).  Defined by: chatpaper.ai "Multi-Head Attention Residuals"
 * abstract.  Reading taken where the page is silent: the key RMSNorm is per
 * head, over the head's d/H channels with that slice of the gain.
 *   src      [n_src][T][d]
 *   queries  [n_q][H][d/H] float, 1 <= n_q <= 8
 *   out      [n_q][T][d] dtype dt; must not overlap src
 *   lse      [n_q][H][T] float or NULL
 * Limits (H > 1): d/H a multiple of 256 (bf16) / 128 (f32) channels; the
 * phase-1 limits apply.
 */
attnres_status_t mhar_fwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                          int64_t d, int64_t H, attnres_dtype_t dt, const float *queries,
                          int64_t n_q, const float *gain, float eps, void *out, float *lse,
                          void *stream);

/*
 * MHAR inside the two-phase Block schedule, phase 2: mhar_fwd over the cached
 * block representations is phase 1 (its lse [n_q][H][T] keeps the state per
 * head); this folds one layer's partial sum into it head by head: head h
 * scores its slice of the partial with its slice of the query, the gain and
 * the RMSNorm, and merges only its own channels,
 *   s_h = w_h . RMSNorm_h(p_h),  M = max(lse_h, s_h),
 *   out_h = (e^{lse_h-M} o_h + e^{s_h-M} p_h) / (e^{lse_h-M} + e^{s_h-M}).
 * H = 1 is attnres_block_phase2_merge.  With f non-NULL the partial is first
 * updated as in attnres_block_phase2_update_merge (partial_out = partial + f)
 * and the merge scores the update.
 * Defined by: chatpaper.ai "Multi-Head Attention Residuals" abstract (per-head
 * softmax, block-diagonal read) with the b-lab.team summary, section 3
 * (Phase 2 merge).
 *   o        [T][d] dtype dt (one query's slice of the MHAR output)
 *   lse      [H][T] float (the matching slice of the MHAR lse)
 *   partial  [T][d] dtype dt or NULL (no update: out = o; update: p = 0)
 *   f, partial_out  NULL, or as attnres_block_phase2_update_merge
 *   query    [H][d/H] float
 *   out      [T][d] dtype dt; may be o itself
 * Limits (H > 1): a head is a whole number of 16-byte vectors (d/H a multiple
 * of 8 bf16 or 4 f32 channels), and the vectors per head are a multiple of 32
 * or a power of two below 32.
 */
attnres_status_t mhar_phase2_merge(const void *o, const float *lse, const void *partial,
                                   const void *f, void *partial_out, int64_t T, int64_t d,
                                   int64_t H, attnres_dtype_t dt, const float *query,
                                   const float *gain, float eps, void *out, void *stream);

/*
 * Backward of the depth read (Full AttnRes: n_q = 1; a Block layer: its
 * sources [b_0..b_{n-1}, partial]; the queries of a block read together):
 * given the gradients dout of the outputs h_q = sum_i alpha_qi v_i, returns
 * the gradients of the sources, the pseudo-queries and the RMSNorm gain.
 * The weights alpha are recomputed from the sources (nothing is saved by the
 * forward).  Defined by the read of the b-lab.team summary, section 1
 * (h = sum_i alpha_i v_i, alpha = softmax of w . RMSNorm(v_i)), differentiated
 * term by term:
 *   ds_qi = alpha_qi (dout_q . v_i - sum_j alpha_qj dout_q . v_j)
 *   dv_i  = sum_q alpha_qi dout_q + sum_q ds_qi (w_q * g) / r_i
 *           - v_i sum_q ds_qi ((w_q * g) . v_i) / (d r_i^3)
 *   dw_q  = g * sum_{t,i} ds_qi v_i / r_i,   dgain = sum_{t,i,q} ds_qi w_q * v_i / r_i
 * with r_i = sqrt(mean(v_i^2) + eps) (a zero source with eps = 0 passes
 * nothing back through its score).
 *   src        [n_src][T][d], sources src_stride elements apart
 *   queries    [n_q][d] float, n_q >= 1;  gain [d] float or NULL
 *   dout       [n_q][T][d] dtype dt
 *   dsrc       [n_src][T][d] dtype dt, sources dsrc_stride (>= T*d) elements
 *              apart; overwritten, or added to when accumulate = 1 (so the
 *              gradients of several reads of the same sources can be summed)
 *   dqueries   [n_q][d] float, overwritten
 *   dgain      [d] float or NULL, overwritten
 *   workspace  device scratch of at least the size attnres_read_bwd_workspace_size
 *              reports (16-byte aligned), owned by the caller; the sums over
 *              the tokens go through it and are reduced in a fixed order, so
 *              results are bitwise reproducible
 * No output may overlap an input or the workspace.  T = 0 zeroes dqueries and
 * dgain.  The queries are taken in passes over the sources (up to 4 per pass
 * with at most 8 sources, else 2, and 1 with more than 8 sources); later
 * passes add into dsrc and dgain, so with more than one pass a bf16 dsrc is
 * rounded once per pass.  A pass of 3 or 4 queries over at most 8 bf16
 * sources at d = 2048 or 4096 runs as two kernels: the first takes each
 * token's row sums on the tensor cores and writes the token's coefficients
 * (alpha_qi, ds_qi / r_i and the v_i term, 72 floats) to the workspace, the
 * second forms dsrc and the sums over the tokens in slices of channels.  It
 * reads the sources and dout twice and rounds a bf16 dsrc once.  Other
 * passes of 3 or 4 queries run two groups of two in one kernel, the second
 * group adding into the bf16 dsrc the first has rounded.  A pass of one query
 * over 3 to 16 bf16 sources at d = 2048 or 4096 (src and src_stride 16-byte
 * aligned) reads them once through a ring of half-row stages, one CTA per
 * SM, with one partial of the sums over the tokens per CTA.
 * More than 16 sources (Full AttnRes past layer 16): with one query, bf16,
 * at most 64 sources and d = 2048 or 4096, two kernels (the first streams
 * every source once and writes each token's coefficients, 72 floats per
 * chunk of 8 sources, to the workspace; the second forms dsrc and the sums
 * over the tokens in slices of channels).  Otherwise the sources are taken in
 * chunks of 8.  Each chunk's read state (o_c, lse_c) is recomputed, and the
 * backward of the states' online-softmax merge (b-lab.team summary, section
 * 3: LSE = log sum_c e^{lse_c}, beta_c = e^{lse_c - LSE}, h = sum_c beta_c o_c)
 * gives d o_c = beta_c dout and d lse_c = beta_c (dout . o_c - dout . h).
 * Then each chunk runs this backward with its lse gradient
 * (attnres_block_phase1_bwd).  The states are held in dtype dt, so with bf16
 * the query and gain gradients carry that rounding; the workspace then also
 * holds the states (about 2 ceil(n_src/8) n_q T d elements of dt).
 * Limits: at most 256 sources (32 chunks) and, above 16 sources, 8 queries;
 * up to 16 sources, outside the ring form, the n_src + (queries of a pass)
 * rows of a token tile must fit two shared-memory stages (for d = 4096 bf16,
 * n_src + 2 <= 13).
 */
attnres_status_t attnres_read_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                  int64_t d, attnres_dtype_t dt, const float *queries, int64_t n_q,
                                  const float *gain, float eps, const void *dout, void *dsrc,
                                  int64_t dsrc_stride, int accumulate, float *dqueries,
                                  float *dgain, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Workspace bytes attnres_read_bwd needs for these sizes on the current
 * device (an upper bound: partial rows of d floats per query of a pass, one
 * for every token row a CTA holds, one CTA per SM, or one per token range of
 * the two-kernel form; for that form also 72 floats per token and head, so
 * the size grows with T).  No device work is done.
 */
attnres_status_t attnres_read_bwd_workspace_size(int64_t n_src, int64_t T, int64_t d, int64_t n_q,
                                                attnres_dtype_t dt, size_t *bytes);

/*
 * attnres_read_bwd without a caller workspace.  The pages have no counterpart
 * to this entry point.  It serves callers that cannot hand this library device
 * memory: a runtime that reserves its whole device-memory budget up front and
 * hands it out from its own pool, or code that may not call cudaMalloc or
 * cudaFree on its hot path (those calls can synchronize the device, and can
 * fail in the middle of a step).  The backward is attnres_read_bwd's, with its
 * sums over the tokens reduced through a fixed scratch array of 8 MB that the
 * library's image places in device memory (a file-scope __device__ array:
 * every device that loads the library holds it until the process exits).
 * No call allocates or frees memory.
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and keeps it; that first
 * call on each device should come before any stream capture.
 * Limits: a call whose workspace would not fit in the array runs its queries
 * in passes of two, then of one; if even one query per pass does not fit it
 * returns ATTNRES_ERR_UNSUPPORTED.  Every other argument, limit and error is
 * attnres_read_bwd's.
 * Sharing: all calls on a device use the same array, which keeps what the
 * last call left in it; each call writes every scratch value before reading
 * it, so nothing needs clearing.  Calls that overlap on the GPU (on streams
 * that do not wait for each other) race on the array and give wrong results:
 * order them on one stream, or make the streams wait for each other.
 */
attnres_status_t attnres_read_bwd_noalloc(const void *src, int64_t n_src, int64_t src_stride,
                                          int64_t T, int64_t d, attnres_dtype_t dt,
                                          const float *queries, int64_t n_q, const float *gain,
                                          float eps, const void *dout, void *dsrc,
                                          int64_t dsrc_stride, int accumulate, float *dqueries,
                                          float *dgain, void *stream);

/*
 * Backward of Block phase 1 (attnres_block_phase1), whose outputs are the
 * reads o_q and their log-sum-exp lse_q = log sum_i exp(s_qi): the gradients
 * d_o of o and d_lse of lse (the phase-1 state's gradients, as the phase-2
 * merge's backward returns them) give the sources', the queries' and the
 * gain's gradients.  Since d lse_q / d s_qi = alpha_qi, the lse gradient adds
 * alpha_qi d_lse_q to ds_qi of attnres_read_bwd's formula.  Defined by the
 * b-lab.team summary, section 3 (Inference): phase 1 keeps (o, lse) per query.
 *   d_o     [n_q][T][d] dtype dt;  d_lse [n_q][T] float, or NULL (zero)
 * Every other argument, the workspace (attnres_read_bwd_workspace_size) and
 * the limits are attnres_read_bwd's.
 */
attnres_status_t attnres_block_phase1_bwd(const void *src, int64_t n_src, int64_t src_stride,
                                          int64_t T, int64_t d, attnres_dtype_t dt,
                                          const float *queries, int64_t n_q, const float *gain,
                                          float eps, const void *d_o, const float *d_lse, void *dsrc,
                                          int64_t dsrc_stride, int accumulate, float *dqueries,
                                          float *dgain, void *workspace, size_t workspace_bytes,
                                          void *stream);

/*
 * Backward of the phase-2 merge (attnres_block_phase2_merge) for an output
 * gradient dh.  Per token, with r_p = sqrt(mean(p^2) + eps),
 * s_p = (w * g) . p / r_p, a = e^{lse-M} / (e^{lse-M} + e^{s_p-M}), b = 1 - a:
 *   d_o       = a dh
 *   d_lse     = a b (dh . (o - p))
 *   d_partial = b dh - d_lse ((w * g) / r_p - p ((w * g) . p) / (d r_p^3))
 *   dquery    = -g * sum_t d_lse p / r_p,   dgain = -w * sum_t d_lse p / r_p
 * (a zero partial with eps = 0 passes nothing back through its score).
 * Defined by the merge of the b-lab.team summary, section 3 (Inference,
 * Phase 2), differentiated term by term.  partial == NULL (out = o): d_o = dh,
 * d_lse = 0, dquery = dgain = 0, d_partial untouched.
 *   o, partial, dh, d_o, d_partial  [T][d] dtype dt;  lse, d_lse [T] float
 *   query, dquery, dgain            [d] float (dgain may be NULL)
 *   accumulate  1: d_partial += its gradient (the partial sums several layers'
 *               outputs, so their gradients add up); 0: overwritten
 *   workspace   device scratch of attnres_block_phase2_bwd_workspace_size
 *               bytes (16-byte aligned); sums over the tokens go through it
 *               and are reduced in a fixed order (bitwise reproducible)
 * No output may overlap an input, another output or the workspace.
 */
attnres_status_t attnres_block_phase2_bwd(const void *o, const float *lse, const void *partial,
                                          int64_t T, int64_t d, attnres_dtype_t dt,
                                          const float *query, const float *gain, float eps,
                                          const void *dh, void *d_o, float *d_lse, void *d_partial,
                                          int accumulate, float *dquery, float *dgain,
                                          void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes attnres_block_phase2_bwd needs (no device work). */
attnres_status_t attnres_block_phase2_bwd_workspace_size(int64_t T, int64_t d, attnres_dtype_t dt,
                                                        size_t *bytes);

/*
 * Backward of the MHAR read (mhar_fwd): H heads of d/H channels, each head its
 * own read over its slice, so the gradient of head h is attnres_read_bwd's
 * formula on that slice of the sources, output gradients, queries and gain,
 * with d replaced by d/H in the RMS term.  Defined by the chatpaper.ai page
 * "Multi-Head Attention Residuals", abstract (per-head softmax, block-diagonal
 * read, H = 1 is the single-head read; its fused routing kernels serve
 * training, i.e. this backward), with the per-head RMSNorm reading of mhar_fwd.
 *   queries   [n_q][H][d/H] float (the layout mhar_fwd takes)
 *   dqueries  [n_q][H][d/H] float, overwritten
 * Every other argument, the passes over the queries, the workspace and the
 * errors are those of attnres_read_bwd (workspace from
 * mhar_read_bwd_workspace_size).  H = 1 is attnres_read_bwd.  Limits besides
 * attnres_read_bwd's: a head holds a multiple of 32 16-byte vectors (d/H a
 * multiple of 256 channels for bf16, 128 for f32), else
 * ATTNRES_ERR_UNSUPPORTED; d % H != 0 is ATTNRES_ERR_INVALID_ARG.
 */
attnres_status_t mhar_read_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                               int64_t d, int64_t H, attnres_dtype_t dt, const float *queries,
                               int64_t n_q, const float *gain, float eps, const void *dout,
                               void *dsrc, int64_t dsrc_stride, int accumulate, float *dqueries,
                               float *dgain, void *workspace, size_t workspace_bytes,
                               void *stream);

/* Workspace bytes mhar_read_bwd needs (as attnres_read_bwd_workspace_size). */
attnres_status_t mhar_read_bwd_workspace_size(int64_t n_src, int64_t T, int64_t d, int64_t H,
                                             int64_t n_q, attnres_dtype_t dt, size_t *bytes);

/*
 * MSAR, the fused multi-stream depth read for one target layer: every source
 * v_i is expanded into m full-width streams (r = 0 identity; r >= 1 a causal
 * depthwise 1-D convolution along the token axis with kernel size
 * ksizes[r-1]); each stream reads the depth history with its own pseudo-query
 * (its weights sum to 1); the m retrieved states Z^(r) are fused by the H^pre
 * mixer: z = RMSNorm(Flatten(Z)) over m*d, c = sigmoid(z . P), h = sum_r c_r Z^(r).
 * The expanded streams are never written to memory.
 * Defined by: onedev.kr "깊이 방향 어텐션을 다중 스트림으로 확장한 MSAR",
 * sections 무엇과 다른가 (streams, per-stream read, mixer) and 어떻게 쓰나
 * (fused on-demand expansion).  Readings taken: left zero padding, no conv
 * bias, u^(r)[t][c] = sum_{j<k} cw[c][j] v[t-j][c]; Flatten is stream-major
 * (element r*d + c is Z^(r)[c]); plain sigmoid, no bias, no renormalisation.
 *   src       [n_src][T][d]; token 0 is the start of the causal sequence
 *   m         number of streams (must be 4)
 *   ksizes    HOST pointer, m-1 kernel sizes, each 1..16
 *   conv_w    float, kernels packed one after another, kernel r as [d][k_r]
 *   queries   [m][d] float
 *   gain      [d] float or NULL (key RMSNorm gain, shared by the streams)
 *   mix_gain  [m*d] float or NULL (mixer RMSNorm gain)
 *   mix_w     [m*d][m] float (the md x m projection P)
 *   mix_eps   >= 0
 *   out       [T][d] dtype dt; must not overlap src
 * Limits: d <= 4096, d a multiple of 256 (bf16) or 128 (f32) channels
 * divided evenly over a cluster of up to 8 CTAs.
 */
attnres_status_t msar_expand_fwd(const void *src, int64_t n_src, int64_t src_stride,
                                 int64_t T, int64_t d, attnres_dtype_t dt, int64_t m,
                                 const int32_t *ksizes, const float *conv_w,
                                 const float *queries, const float *gain, float eps,
                                 const float *mix_gain, const float *mix_w, float mix_eps,
                                 void *out, void *stream);

/*
 * MSAR for one chunk of a longer sequence (chunked prefill): src holds, per
 * source, T_prev rows that earlier chunks already processed followed by the
 * T rows of this chunk; out receives the T outputs of this chunk.  The
 * causal convolutions read back into the T_prev history rows; rows before
 * the start of src count as zero, so T_prev = max kernel size - 1 (or every
 * earlier token) gives exactly the outputs msar_expand_fwd would give for
 * these tokens over the whole sequence.  T_prev = 0 is msar_expand_fwd.
 * Defined by: onedev.kr MSAR page, sections 무엇과 다른가 and 어떻게 쓰나 (the
 * causal stream expansion, fused on demand), with chunked prefill of long
 * contexts from the dimensionstp.github.io review, sections 3-2 5) and 4-3.
 *   src     [n_src] x [T_prev + T][d], sources src_stride (>= (T_prev+T)*d)
 *           elements apart
 *   out     [T][d] dtype dt; must not overlap src
 * All other arguments, limits and errors are those of msar_expand_fwd;
 * T_prev < 0 is ATTNRES_ERR_INVALID_ARG.
 */
attnres_status_t msar_expand_fwd_chunk(const void *src, int64_t n_src, int64_t src_stride,
                                       int64_t T_prev, int64_t T, int64_t d, attnres_dtype_t dt,
                                       int64_t m, const int32_t *ksizes, const float *conv_w,
                                       const float *queries, const float *gain, float eps,
                                       const float *mix_gain, const float *mix_w, float mix_eps,
                                       void *out, void *stream);

/*
 * msar_expand_fwd with each source's own conv kernels: source i is expanded
 * with the kernels packed (as msar_expand_fwd's conv_w) at
 * conv_w + i * conv_src_stride floats.  Defined by the MSAR page, section
 * 무엇과 다른가 (the streams v_i^(r) of each source), read here with per-source
 * kernels; msar_expand_fwd is the reading in which all sources share them.
 *   conv_src_stride  > 0 floats; at least d * (k_1 + k_2 + k_3) with more than
 *                    one source (else ATTNRES_ERR_INVALID_ARG), and then a
 *                    multiple of 4 (16-byte aligned kernels; else
 *                    ATTNRES_ERR_UNSUPPORTED)
 * Every other argument and limit as msar_expand_fwd.  The kernels of 8
 * sources do not fit in shared memory, so they are read through L2 as the
 * convolution needs them: slower than the shared-kernel read.
 */
attnres_status_t msar_expand_fwd_ps(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                    int64_t d, attnres_dtype_t dt, int64_t m,
                                    const int32_t *ksizes, const float *conv_w,
                                    int64_t conv_src_stride, const float *queries,
                                    const float *gain, float eps, const float *mix_gain,
                                    const float *mix_w, float mix_eps, void *out, void *stream);

/*
 * MSAR inside the two-phase Block schedule, phase 1: the queries of S layers
 * of a block read the completed (cached) sources in one pass.  Every source
 * is expanded once into its m streams (as msar_expand_fwd) and, for every
 * layer s and stream r, the read's state over the sources is kept:
 *   o_s^(r)   = sum_i softmax_i(w_s^(r) . RMSNorm(u_i^(r))) u_i^(r)
 *   lse_s^(r) = log sum_i exp(w_s^(r) . RMSNorm(u_i^(r)))
 * Defined by: onedev.kr "깊이 방향 어텐션을 다중 스트림으로 확장한 MSAR",
 * section 어떻게 쓰나 (AttnRes's caching and two-phase computation carry over:
 * a block's target queries are batched against the completed sources, and
 * each layer then merges its own partial sum with the online softmax), with
 * the phase-1 state of the b-lab.team summary, section 3 (Inference).
 * Reading taken: the streams of a source are the source's own (the page
 * writes them v_i^(r), with no layer index), so one conv_w serves every
 * layer and the partials.
 *   src       [n_src][T][d], n_src <= 8
 *   queries   [S][m][d] float (m = 4 streams per layer)
 *   o         [S][m][T][d] dtype dt;  lse [S][m][T] float
 * Other arguments and limits as msar_expand_fwd.  More than 4 layers are
 * read in groups of 4 (each group expands the sources again).
 */
attnres_status_t msar_block_phase1(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                   int64_t d, attnres_dtype_t dt, int64_t m,
                                   const int32_t *ksizes, const float *conv_w,
                                   const float *queries, int64_t S, const float *gain, float eps,
                                   void *o, float *lse, void *stream);

/*
 * MSAR two-phase, phase 2 of one layer: the layer's partial sum is its one
 * more source.  It is expanded into its m streams with the same kernels
 * (causally over the partial's own history, token 0 first); each stream's
 * score s_p^(r) = w^(r) . RMSNorm(u_p^(r)) is merged into that stream's
 * phase-1 state by the online-softmax merge (b-lab.team summary, section 3,
 * Phase 2):  Z^(r) = (e^{lse-M} o^(r) + e^{s_p-M} u_p^(r)) / (e^{lse-M} + e^{s_p-M});
 * the merged Z go through the H^pre mixer as in msar_expand_fwd.  partial ==
 * NULL (the block's first layer) mixes Z^(r) = o^(r).
 *   o         [m][T][d] dtype dt (layer s of msar_block_phase1's o)
 *   lse       [m][T] float
 *   partial   [T][d] dtype dt, or NULL
 *   query     [m][d] float (the layer's stream queries)
 *   out       [T][d] dtype dt; must not overlap o, lse or partial
 * Other arguments and limits as msar_expand_fwd.
 */
attnres_status_t msar_block_phase2(const void *o, const float *lse, const void *partial, int64_t T,
                                   int64_t d, attnres_dtype_t dt, int64_t m,
                                   const int32_t *ksizes, const float *conv_w, const float *query,
                                   const float *gain, float eps, const float *mix_gain,
                                   const float *mix_w, float mix_eps, void *out, void *stream);

/*
 * Backward of msar_expand_fwd for an output gradient dh: the gradients of the
 * sources, the conv kernels, the stream queries, the key gain and the mixer's
 * gain and projection.  Defined by the chain rule through the three steps of
 * the MSAR page, section 무엇과 다른가 (onedev.kr "깊이 방향 어텐션을 다중
 * 스트림으로 확장한 MSAR"): the H^pre mixer (sigmoid of the RMSNorm'd flat
 * Z times P), each stream's depth read (the backward of attnres_read_bwd,
 * one query per stream), and the causal depthwise convolutions, whose
 * transpose sends du^(r)[t] back to the rows t-j it read.  Readings as
 * msar_expand_fwd.
 *   src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, queries, gain, eps,
 *   mix_gain, mix_w, mix_eps   as msar_expand_fwd (the forward's inputs)
 *   dh         [T][d] dtype dt
 *   dsrc       [n_src] x [T][d] dtype dt, dsrc_stride (>= T*d) elements
 *              apart; overwritten; must not overlap src or dh
 *   dconv_w    float, packed as conv_w; overwritten
 *   dqueries   [m][d] float; overwritten
 *   dgain      [d] float or NULL (the gain's gradient, summed over the
 *              streams; with gain NULL it is the gradient at an all-ones gain)
 *   dmix_gain  [m*d] float or NULL (same convention); dmix_w [m*d][m] float
 *   workspace  device scratch of msar_expand_bwd_workspace_size bytes (it
 *              holds the conv streams, the per-stream reads and their
 *              gradients: about (7 n_src + 8) T d elements of dtype dt);
 *              must not overlap any other argument
 * The parameter gradients are sums over the tokens taken in a fixed order
 * (same inputs, same bits).  The streams, the per-stream reads and their
 * gradients are held in dtype dt.  T = 0 zeroes the parameter gradients.
 * Limits: m = 4, kernel sizes 1..16, d = 1024, 2048 or 4096, n_src <= 16,
 * else ATTNRES_ERR_UNSUPPORTED; pointers 16-byte aligned except the float
 * gradients dconv_w, dqueries, dgain, dmix_gain (4-byte).  A NULL required
 * pointer, a short workspace or overlapping outputs is
 * ATTNRES_ERR_INVALID_ARG.
 */
attnres_status_t msar_expand_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                 int64_t d, attnres_dtype_t dt, int64_t m, const int32_t *ksizes,
                                 const float *conv_w, const float *queries, const float *gain,
                                 float eps, const float *mix_gain, const float *mix_w, float mix_eps,
                                 const void *dh, void *dsrc, int64_t dsrc_stride, float *dconv_w,
                                 float *dqueries, float *dgain, float *dmix_gain, float *dmix_w,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * msar_expand_bwd for msar_expand_fwd_ps (each source's own conv kernels):
 * source i's kernels are read at conv_w + i * conv_src_stride and its kernel
 * gradient is written at dconv_w + i * conv_src_stride (packed as its
 * kernels; the floats between one source's set and the next are not
 * written).  Defined by the same chain rule as msar_expand_bwd, with source
 * i's streams taken through its own kernels (MSAR page, section 무엇과 다른가,
 * the streams v_i^(r) of each source).
 *   conv_src_stride  > 0 floats; at least d * (k_1 + k_2 + k_3) with more than
 *                    one source (else ATTNRES_ERR_INVALID_ARG), and then a
 *                    multiple of 4 (else ATTNRES_ERR_UNSUPPORTED)
 *   dconv_w          float, n_src sets conv_src_stride apart; overwritten
 * Every other argument, the workspace (msar_expand_bwd_workspace_size) and the
 * limits are msar_expand_bwd's.
 */
attnres_status_t msar_expand_bwd_ps(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                    int64_t d, attnres_dtype_t dt, int64_t m, const int32_t *ksizes,
                                    const float *conv_w, int64_t conv_src_stride, const float *queries,
                                    const float *gain, float eps, const float *mix_gain,
                                    const float *mix_w, float mix_eps, const void *dh, void *dsrc,
                                    int64_t dsrc_stride, float *dconv_w, float *dqueries, float *dgain,
                                    float *dmix_gain, float *dmix_w, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * msar_expand_bwd over one chunk of a longer sequence, so that the workspace
 * is sized by the chunk's tokens, not the sequence's: the backward of the
 * chunked prefill msar_expand_fwd_chunk.  src holds, per source, T_prev
 * history rows followed by the chunk's T rows (as msar_expand_fwd_chunk); dh
 * is the chunk's [T][d].  The causal convolutions read back into the history
 * rows, so their transpose sends part of the chunk's gradient there.
 * Defined by the chain rule of msar_expand_bwd (MSAR page, section 무엇과
 * 다른가) over the chunk, with the chunked prefill of the dimensionstp.github.io
 * review, sections 3-2 5) and 4-3.
 *   src        [n_src] x [T_prev + T][d], src_stride (>= (T_prev+T)*d) apart
 *   dsrc       [n_src] x [T_prev + T][d], dsrc_stride apart: the chunk's T
 *              rows are overwritten; the chunk's share of the gradient of
 *              the T_prev history rows is ADDED into the first T_prev rows
 *   accumulate 0: the parameter gradients (dconv_w, dqueries, dgain,
 *              dmix_gain, dmix_w) are overwritten; 1: the chunk's sums are
 *              added into them
 *   workspace  msar_expand_bwd_workspace_size(n_src, T, ...) bytes
 * A whole sequence in order: chunk c of rows [t_c, t_{c+1}) with
 * T_prev = min(t_c, max kernel size - 1) (src and dsrc pointing T_prev rows
 * before t_c), accumulate = 0 for the first chunk and 1 after; then dsrc and
 * every parameter gradient equal msar_expand_bwd's over the whole sequence
 * (up to the order of the sums and one more rounding of the T_prev rows).
 * Chunks must run in increasing order on one stream: a chunk overwrites its
 * own rows, and the next chunk adds into their last T_prev.
 * Every other argument, limit and error is msar_expand_bwd's; T_prev < 0 or
 * accumulate not 0 or 1 is ATTNRES_ERR_INVALID_ARG.
 */
attnres_status_t msar_expand_bwd_chunk(const void *src, int64_t n_src, int64_t src_stride,
                                       int64_t T_prev, int64_t T, int64_t d, attnres_dtype_t dt,
                                       int64_t m, const int32_t *ksizes, const float *conv_w,
                                       const float *queries, const float *gain, float eps,
                                       const float *mix_gain, const float *mix_w, float mix_eps,
                                       const void *dh, void *dsrc, int64_t dsrc_stride,
                                       int accumulate, float *dconv_w, float *dqueries,
                                       float *dgain, float *dmix_gain, float *dmix_w,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes msar_expand_bwd (and msar_expand_bwd_ps) needs for these
 * sizes on the current device. */
attnres_status_t msar_expand_bwd_workspace_size(int64_t n_src, int64_t T, int64_t d,
                                               attnres_dtype_t dt, int64_t m,
                                               const int32_t *ksizes, size_t *bytes);

/*
 * msar_expand_fwd with a caller workspace: the same read as a chain that
 * writes the conv streams once, reads each stream with the forward read
 * kernels and mixes the per-stream reads.  The fused msar_expand_fwd never
 * writes a stream (the pages' on-demand expansion, MSAR page, section 어떻게
 * 쓰나) but synchronises a cluster of CTAs per token; on GB300 the chain is
 * faster where the memory for it is available.  The per-stream reads are
 * held in dtype dt before the mixer (the fused read keeps them in fp32), so
 * bf16 results differ from msar_expand_fwd's within the bf16 tolerance.
 *   conv_src_stride  0: one set of kernels for every source (msar_expand_fwd);
 *                    > 0: source i's kernels at conv_w + i * conv_src_stride
 *                    (msar_expand_fwd_ps; >= d * (k_1 + k_2 + k_3) with more
 *                    than one source, else ATTNRES_ERR_INVALID_ARG)
 *   workspace        device scratch of msar_expand_fwd_ws_workspace_size bytes
 *                    (the streams and the per-stream reads: (3 n_src + 4) T d
 *                    elements of dtype dt and T d / 1024 x 9 floats); must not
 *                    overlap src or out
 * Every other argument as msar_expand_fwd.  Limits: m = 4, kernel sizes
 * 1..16, d a multiple of 1024 up to 16384 (else ATTNRES_ERR_UNSUPPORTED);
 * queries, mix_w, gain, out and workspace 16-byte aligned, conv_w and
 * mix_gain 4-byte.
 */
attnres_status_t msar_expand_fwd_ws(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                    int64_t d, attnres_dtype_t dt, int64_t m, const int32_t *ksizes,
                                    const float *conv_w, int64_t conv_src_stride, const float *queries,
                                    const float *gain, float eps, const float *mix_gain,
                                    const float *mix_w, float mix_eps, void *out, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* Workspace bytes msar_expand_fwd_ws needs for these sizes. */
attnres_status_t msar_expand_fwd_ws_workspace_size(int64_t n_src, int64_t T, int64_t d,
                                                  attnres_dtype_t dt, size_t *bytes);

/*
 * msar_block_phase1 with a caller workspace: every cached source's three conv
 * streams are written once, then each stream (the sources themselves for
 * stream 0) is read by that stream's queries of all S layers with the
 * forward read kernels (up to 8 layers per launch), giving the same state o,
 * lse in the same layout.  The streams are held in dtype dt before the read
 * (the fused phase 1 keeps them in fp32).
 *   workspace  device scratch of msar_block_phase1_ws_workspace_size bytes
 *              (the streams: 3 n_src T d elements of dtype dt, plus the
 *              queries regrouped by stream and one group's lse); must not
 *              overlap src, o or lse
 * Every other argument as msar_block_phase1, without its n_src <= 8 limit.
 * Limits: d a multiple of 512 up to 16384 (else ATTNRES_ERR_UNSUPPORTED).
 */
attnres_status_t msar_block_phase1_ws(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                      int64_t d, attnres_dtype_t dt, int64_t m,
                                      const int32_t *ksizes, const float *conv_w,
                                      const float *queries, int64_t S, const float *gain, float eps,
                                      void *o, float *lse, void *workspace, size_t workspace_bytes,
                                      void *stream);

/* Workspace bytes msar_block_phase1_ws needs for these sizes. */
attnres_status_t msar_block_phase1_ws_workspace_size(int64_t n_src, int64_t T, int64_t d,
                                                    attnres_dtype_t dt, int64_t S, size_t *bytes);

/*
 * msar_block_phase2 with a caller workspace: the partial's three conv streams
 * are written once, each stream of the partial is merged into that stream's
 * phase-1 state by the Block merge (attnres_block_phase2_merge's kernel, one
 * launch per stream) and the merged streams Z^(r) go through the mixer as in
 * msar_expand_fwd_ws.  partial == NULL mixes Z^(r) = o^(r).  The streams and
 * the merged Z are held in dtype dt (the fused phase 2 keeps them in fp32).
 *   workspace  device scratch of msar_block_phase2_ws_workspace_size bytes
 *              (7 T d elements of dtype dt and T d / 1024 x 9 floats); must
 *              not overlap o, lse, partial or out
 * Every other argument as msar_block_phase2.  Limits: d a multiple of 1024 up
 * to 16384 (else ATTNRES_ERR_UNSUPPORTED).
 */
attnres_status_t msar_block_phase2_ws(const void *o, const float *lse, const void *partial, int64_t T,
                                      int64_t d, attnres_dtype_t dt, int64_t m,
                                      const int32_t *ksizes, const float *conv_w, const float *query,
                                      const float *gain, float eps, const float *mix_gain,
                                      const float *mix_w, float mix_eps, void *out, void *workspace,
                                      size_t workspace_bytes, void *stream);

/* Workspace bytes msar_block_phase2_ws needs for these sizes. */
attnres_status_t msar_block_phase2_ws_workspace_size(int64_t T, int64_t d, attnres_dtype_t dt,
                                                    size_t *bytes);

/*
 * Backward of msar_block_phase2 (one layer of MSAR's two-phase schedule) for
 * an output gradient dh.  Defined by the chain rule through phase 2's steps:
 * the H^pre mixer over the merged streams (as msar_expand_bwd), each stream's
 * online-softmax merge (b-lab.team summary, section 3, Phase 2; backward as
 * attnres_block_phase2_bwd, the partial's stream r being that merge's partial
 * and w^(r) its query), and the partial's causal convolutions (MSAR page,
 * sections 무엇과 다른가 and 어떻게 쓰나).  Together with msar_block_phase1_bwd
 * it equals msar_expand_bwd over [cached sources, partial].
 *   o, lse, partial, T, d, dt, m, ksizes, conv_w, query, gain, eps, mix_gain,
 *   mix_w, mix_eps   as msar_block_phase2 (the forward's inputs)
 *   dh         [T][d] dtype dt
 *   d_o        [m][T][d] dtype dt; d_lse [m][T] float: the gradients of the
 *              phase-1 state (to msar_block_phase1_bwd); overwritten
 *   d_partial  [T][d] dtype dt (required with a partial; NULL otherwise)
 *   dconv_w    float, packed as conv_w: the partial's share (zero without one)
 *   dquery     [m][d] float: the merges' share; dgain [d] float or NULL (the
 *              merges' share); dmix_gain [m*d] or NULL, dmix_w [m*d][m]
 *   workspace  device scratch of msar_block_phase2_bwd_workspace_size bytes
 * All outputs are overwritten; parameter sums over tokens are in a fixed
 * order.  Limits: m = 4, kernel sizes 1..16, d = 1024, 2048 or 4096 (else
 * ATTNRES_ERR_UNSUPPORTED).  Overlapping outputs, or outputs overlapping the
 * inputs or the workspace, are ATTNRES_ERR_INVALID_ARG.
 */
attnres_status_t msar_block_phase2_bwd(const void *o, const float *lse, const void *partial, int64_t T,
                                       int64_t d, attnres_dtype_t dt, int64_t m,
                                       const int32_t *ksizes, const float *conv_w, const float *query,
                                       const float *gain, float eps, const float *mix_gain,
                                       const float *mix_w, float mix_eps, const void *dh, void *d_o,
                                       float *d_lse, void *d_partial, float *dconv_w, float *dquery,
                                       float *dgain, float *dmix_gain, float *dmix_w, void *workspace,
                                       size_t workspace_bytes, void *stream);

/* Workspace bytes msar_block_phase2_bwd needs for these sizes on the current device. */
attnres_status_t msar_block_phase2_bwd_workspace_size(int64_t T, int64_t d, attnres_dtype_t dt, int64_t m,
                                                     const int32_t *ksizes, size_t *bytes);

/*
 * Backward of msar_block_phase1 for gradients d_o [S][m][T][d] and d_lse
 * [S][m][T] of its state (the sums of every layer's msar_block_phase2_bwd
 * d_o and d_lse for the block).  Defined by the chain rule through phase 1:
 * each stream's read of the cached sources' streams by the S layers' queries,
 * with its log-sum-exp (attnres_block_phase1_bwd's formula), and the causal
 * convolutions (MSAR page, section 무엇과 다른가; b-lab.team summary, section 3).
 *   src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, queries, S, gain,
 *   eps        as msar_block_phase1
 *   dsrc       [n_src] x [T][d] dtype dt, dsrc_stride apart; overwritten
 *   dconv_w    float, packed as conv_w (the cached sources' share)
 *   dqueries   [S][m][d] float (phase 1's share); dgain [d] float or NULL
 *   workspace  device scratch of msar_block_phase1_bwd_workspace_size bytes
 * Limits: m = 4, kernel sizes 1..16, d a multiple of 512 up to 4096, n_src <=
 * 16 (else ATTNRES_ERR_UNSUPPORTED); errors otherwise as msar_expand_bwd.
 */
attnres_status_t msar_block_phase1_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                       int64_t d, attnres_dtype_t dt, int64_t m,
                                       const int32_t *ksizes, const float *conv_w,
                                       const float *queries, int64_t S, const float *gain, float eps,
                                       const void *d_o, const float *d_lse, void *dsrc,
                                       int64_t dsrc_stride, float *dconv_w, float *dqueries,
                                       float *dgain, void *workspace, size_t workspace_bytes,
                                       void *stream);

/* Workspace bytes msar_block_phase1_bwd needs for these sizes on the current device. */
attnres_status_t msar_block_phase1_bwd_workspace_size(int64_t n_src, int64_t T, int64_t d,
                                                     attnres_dtype_t dt, int64_t m,
                                                     const int32_t *ksizes, int64_t S, size_t *bytes);

/* Static description of a status code (never NULL). */
const char *attnres_status_string(attnres_status_t status);

/* Message of the last CUDA error seen by an entry point on this host thread
 * ("" if none). */
const char *attnres_last_cuda_error(void);

/*
 * Waits for all work on stream, then reports (and clears) a device-side
 * failure recorded by any kernel of this library on the current device since
 * the last call: ATTNRES_ERR_TIMEOUT if a bounded wait inside a kernel ran
 * out of time (that kernel's outputs are invalid), ATTNRES_ERR_CUDA if the
 * synchronisation itself failed, else ATTNRES_OK.
 */
attnres_status_t attnres_sync_status(void *stream);

/*
 * Failure-detection hooks, meant for tests.
 * attnres_debug_set_wait_timeout_ns: limit of every device-side wait, in
 *   nanoseconds (default 2e9; 0 restores the default).
 * attnres_debug_set_stall_injection: when nonzero, kernels that stage data
 *   with bulk copies issue no copies, so their first wait can only end by
 *   running out of time; they then record ATTNRES_ERR_TIMEOUT and return
 *   without touching memory.  Applies to launches made after the call.
 */
void attnres_debug_set_wait_timeout_ns(uint64_t ns);
void attnres_debug_set_stall_injection(int enable);

/*
 * Kernel selection, meant for tests and measurements: 0 (default) lets the
 * library pick (for one head and at most 64 tokens the few-token kernel, a
 * token per cluster of CTAs, when it applies; else tensor-core kernels for
 * bf16 reads with <= 4 queries at d = 1024, 2048 or 4096 and <= 8 sources,
 * and at d = 4096 for more sources where the chunked tensor-core kernel was
 * measured faster; the general CUDA-core kernel otherwise); 1 forces the
 * general kernel for Full / phase 1 / MHAR; 2 takes the tensor-core kernels
 * wherever they apply (the chunked one for any source count > 8 at d = 4096);
 * 3 takes the few-token kernel wherever it applies (one head, <= 16 sources
 * with <= 2 queries or <= 8 with 4, any number of tokens).  All compute the
 * same operation.  Applies to calls made afterwards; other values act as 0.
 */
void attnres_debug_set_kernel_variant(int variant);

/* Library version string, e.g. "attnres 0.1.0 sm_103a". */
const char *attnres_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_H */
