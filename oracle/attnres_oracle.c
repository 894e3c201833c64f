/*
 * attnres_oracle.c -- plain, slow, single-threaded CPU oracle for the
 * Attention Residuals depth-wise softmax read.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library.
 *
 * Every function works in IEEE double precision on the exact input values
 * (bf16 inputs are widened exactly before they get here).  No blocking, no
 * fusion, no reordering beyond what the definitions state; loops follow the
 * formulas term by term so they can be checked against the pages by eye.
 *
 * Page labels used in the citations below:
 *   [Summary]   b-lab.team summary of "Attention Residuals"
 *               (sections 1 Full AttnRes, 2 Block AttnRes, 3 Infrastructure)
 *   [Review]    dimensionstp.github.io "Attention Residuals" review
 *               (sections 2-2, 3-2, 4-3)
 *   [Tutorial]  ai-systems-engineering.com "Attention Residuals: 지나온 층의
 *               출력을 선택해서 읽기" (Figs. 2-4 and their worked example)
 *   [MSAR]      onedev.kr "깊이 방향 어텐션을 다중 스트림으로 확장한 MSAR"
 *               (sections 무엇과 다른가, 어떻게 쓰나)
 *   [MHAR]      chatpaper.ai "Multi-Head Attention Residuals" abstract
 *
 * Layouts (row-major, contiguous):
 *   sources   src[n_src][T][d]
 *   queries   w[n_q][d]          (MHAR: w[n_q][H][d/H])
 *   gain      g[d] or NULL (NULL means every channel has gain 1)
 *
 * Return value: 0 on success, -1 on an invalid argument.
 *
 * Parity status: every exported function below is pinned by the non-GPU
 * tests (worked example, closed forms, invariants, brute force); none is
 * "parity unpinned".
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* Building blocks                                                          */
/* ---------------------------------------------------------------------- */

/* RMSNorm of one vector, [Summary §1] kernel phi(q,k) = exp(q^T RMSNorm(k)),
 * [Tutorial Fig. 3] "gain 1, epsilon omitted": y = g * x / sqrt(mean(x^2)+eps).
 * Reading taken where the pages are silent: eps sits inside the square root,
 * added to the mean square; a zero vector with eps = 0 normalises to zero. */
static void rmsnorm(const double *x, const double *g, int64_t n, double eps,
                    double *y)
{
    double ms = 0.0;
    for (int64_t c = 0; c < n; ++c) ms += x[c] * x[c];
    ms /= (double)n;
    double denom = sqrt(ms + eps);
    for (int64_t c = 0; c < n; ++c) {
        double gc = g ? g[c] : 1.0;
        y[c] = (denom > 0.0) ? gc * x[c] / denom : 0.0;
    }
}

/* score = w^T RMSNorm(k)  [Summary §1], [Review §2-2 eq. for alpha] */
static double score(const double *w, const double *k, const double *g,
                    int64_t n, double eps, double *tmp)
{
    rmsnorm(k, g, n, eps, tmp);
    double s = 0.0;
    for (int64_t c = 0; c < n; ++c) s += w[c] * tmp[c];
    return s;
}

/* softmax over depth: alpha_i = exp(s_i - max) / sum_j exp(s_j - max);
 * also returns lse = max + log(sum_j exp(s_j - max)).  [Summary §1 alpha] */
static double softmax(const double *s, int64_t n, double *alpha)
{
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) if (s[i] > m) m = s[i];
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) { alpha[i] = exp(s[i] - m); l += alpha[i]; }
    for (int64_t i = 0; i < n; ++i) alpha[i] /= l;
    return m + log(l);
}

/* One depth read for one token over a list of source rows:
 *   h = sum_i alpha_i v_i  with  alpha = softmax_i(w^T RMSNorm(v_i)).
 * The weighted sum uses the raw (un-normalised) values: [Tutorial Fig. 3]
 * "the sqrt(3) used for the score is not multiplied back onto the source".
 * rows[i] points at v_i (length n).  alpha_out/lse_out may be NULL. */
static int read_one(const double *const *rows, int64_t n_src, int64_t n,
                    const double *w, const double *g, double eps,
                    double *h, double *alpha_out, double *lse_out)
{
    double *tmp = (double *)malloc(sizeof(double) * (size_t)n);
    double *s = (double *)malloc(sizeof(double) * (size_t)n_src);
    double *a = (double *)malloc(sizeof(double) * (size_t)n_src);
    if (!tmp || !s || !a) { free(tmp); free(s); free(a); return -1; }
    for (int64_t i = 0; i < n_src; ++i) s[i] = score(w, rows[i], g, n, eps, tmp);
    double lse = softmax(s, n_src, a);
    for (int64_t c = 0; c < n; ++c) {
        double acc = 0.0;
        for (int64_t i = 0; i < n_src; ++i) acc += a[i] * rows[i][c];
        h[c] = acc;
    }
    if (alpha_out) for (int64_t i = 0; i < n_src; ++i) alpha_out[i] = a[i];
    if (lse_out) *lse_out = lse;
    free(tmp); free(s); free(a);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Full AttnRes                                                            */
/* ---------------------------------------------------------------------- */

/* Full AttnRes read for one layer, [Summary §1] h_l = sum_{i<l} alpha_{i->l} v_i,
 * [Review §3-2 1)].  src[n_src][T][d] are the sources v_0..v_{n_src-1};
 * out[T][d]; lse[T] (may be NULL) = log sum_i exp(score_i); alpha[T][n_src]
 * (may be NULL) receives the weights. */
int oracle_full(const double *src, int64_t n_src, int64_t T, int64_t d,
                const double *query, const double *gain, double eps,
                double *out, double *lse, double *alpha)
{
    if (!src || !query || !out || n_src < 1 || T < 0 || d < 1 || eps < 0) return -1;
    const double **rows = (const double **)malloc(sizeof(double *) * (size_t)n_src);
    if (!rows) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < n_src; ++i) rows[i] = src + (i * T + t) * d;
        if (read_one(rows, n_src, d, query, gain, eps, out + t * d,
                     alpha ? alpha + t * n_src : NULL, lse ? lse + t : NULL)) {
            free(rows); return -1;
        }
    }
    free(rows);
    return 0;
}

/* The weighted sum alone with given weights: h[t] = sum_i alpha[t][i] v_i[t].
 * [Tutorial Fig. 2] table "each weight multiplies the whole source vector". */
int oracle_weighted_sum(const double *src, int64_t n_src, int64_t T, int64_t d,
                        const double *alpha, double *out)
{
    if (!src || !alpha || !out || n_src < 1 || T < 0 || d < 1) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t i = 0; i < n_src; ++i) acc += alpha[t * n_src + i] * src[(i * T + t) * d + c];
            out[t * d + c] = acc;
        }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Block AttnRes                                                           */
/* ---------------------------------------------------------------------- */

/* Block AttnRes, one block, computed one layer at a time ("one-shot").
 * [Summary §2] value matrix of layer i of block n:
 *   i = 1:  [b_0, ..., b_{n-1}]
 *   i >= 2: [b_0, ..., b_{n-1}, b^{(n)}_{i-1}]   (current partial sum)
 * [Tutorial Fig. 4]: the first sublayer of a block does not read the empty
 * current sum.  cache[N][T][d] holds b_0..b_{N-1}; partials[S][T][d] holds
 * the partial sum read by each layer (slot 0 is ignored: layer 1 has none);
 * queries[S][d]; out[S][T][d]. */
int oracle_block_oneshot(const double *cache, int64_t N, const double *partials,
                         int64_t S, int64_t T, int64_t d, const double *queries,
                         const double *gain, double eps, double *out)
{
    if (!cache || !queries || !out || N < 1 || S < 1 || T < 0 || d < 1 || eps < 0) return -1;
    if (S > 1 && !partials) return -1;
    const double **rows = (const double **)malloc(sizeof(double *) * (size_t)(N + 1));
    if (!rows) return -1;
    for (int64_t li = 0; li < S; ++li) {          /* li = i - 1 */
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t n = 0; n < N; ++n) rows[n] = cache + (n * T + t) * d;
            int64_t n_src = N;
            if (li >= 1) { rows[N] = partials + (li * T + t) * d; n_src = N + 1; }
            if (read_one(rows, n_src, d, queries + li * d, gain, eps,
                         out + (li * T + t) * d, NULL, NULL)) { free(rows); return -1; }
        }
    }
    free(rows);
    return 0;
}

/* Phase 1 of the two-phase schedule, [Summary §3 Inference, Phase 1],
 * [Review §3-2 4)]: all n_q queries of a block read the N cached block
 * representations; keeps the softmax state normalised as
 *   o_q = acc_q / l_q   and   lse_q = m_q + log l_q.
 * o[n_q][T][d], lse[n_q][T]. */
int oracle_block_phase1(const double *cache, int64_t N, int64_t T, int64_t d,
                        const double *queries, int64_t n_q, const double *gain,
                        double eps, double *o, double *lse)
{
    if (!cache || !queries || !o || !lse || N < 1 || n_q < 1 || T < 0 || d < 1 || eps < 0) return -1;
    for (int64_t q = 0; q < n_q; ++q)
        if (oracle_full(cache, N, T, d, queries + q * d, gain, eps,
                        o + q * T * d, lse + q * T, NULL)) return -1;
    return 0;
}

/* Phase 2 of the two-phase schedule, [Summary §3 Inference, Phase 2],
 * [Review §3-2 4) "online softmax merge"]: fold the score of the current
 * partial sum p into the phase-1 state (o, lse):
 *   s_p = w^T RMSNorm(p),  M = max(lse, s_p),
 *   h = (e^{lse-M} o + e^{s_p-M} p) / (e^{lse-M} + e^{s_p-M}).
 * partial == NULL (first layer of the block) gives h = o. */
int oracle_block_phase2(const double *o, const double *lse, const double *partial,
                        int64_t T, int64_t d, const double *query,
                        const double *gain, double eps, double *out)
{
    if (!o || !lse || !query || !out || T < 0 || d < 1 || eps < 0) return -1;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)d);
    if (!tmp) return -1;
    for (int64_t t = 0; t < T; ++t) {
        const double *ot = o + t * d;
        if (!partial) { for (int64_t c = 0; c < d; ++c) out[t * d + c] = ot[c]; continue; }
        const double *pt = partial + t * d;
        double sp = score(query, pt, gain, d, eps, tmp);
        double M = lse[t] > sp ? lse[t] : sp;
        double a = exp(lse[t] - M), b = exp(sp - M);
        for (int64_t c = 0; c < d; ++c) out[t * d + c] = (a * ot[c] + b * pt[c]) / (a + b);
    }
    free(tmp);
    return 0;
}

/* Intra-block partial-sum update fused with the next layer's merge.
 * [Summary §2 Block AttnRes]: the current block's source for layer i >= 2 is
 * the partial sum b_{i-1}^(n) of the block's layer outputs so far;
 * [Tutorial Fig. 4]: once a layer's output f is produced, only the current
 * partial sum changes, to the old partial plus f (the embedding and the
 * completed block sums stay as they are).  [Summary §3 Inference, Phase 2]:
 * the merge of the next layer then scores that new partial.
 *   p_out = p + f            (p == NULL: the block's first output, p_out = f)
 *   out   = phase-2 merge of (o, lse) with p_out      (oracle_block_phase2)
 * p, f, p_out, o, out [T][d]; lse [T]. */
int oracle_block_phase2_update(const double *p, const double *f, const double *o,
                               const double *lse, int64_t T, int64_t d, const double *query,
                               const double *gain, double eps, double *p_out, double *out)
{
    if (!f || !o || !lse || !query || !p_out || !out || T < 0 || d < 1 || eps < 0) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < d; ++c)
            p_out[t * d + c] = (p ? p[t * d + c] : 0.0) + f[t * d + c];
    return oracle_block_phase2(o, lse, p_out, T, d, query, gain, eps, out);
}

/* ---------------------------------------------------------------------- */
/* Backward of the read                                                     */
/* ---------------------------------------------------------------------- */

/* Gradients of the depth read of n_q queries over n_src sources (Full
 * AttnRes: n_q = 1; a Block layer: its sources [b_0..b_{n-1}, partial]; Block
 * phase 1: the block's S queries) for a loss whose gradient with respect to
 * every output h_q[t] is dout[q][t] (the backward of [Summary §1]; the
 * forward is read_one, so alpha is recomputed from the sources).  The chain
 * rule is taken step by step, per token:
 *   forward  r_i = sqrt(mean(v_i^2) + eps),  k_i = g * v_i / r_i,
 *            s_qi = w_q . k_i,  alpha_q = softmax_i(s_q),  h_q = sum_i alpha_qi v_i
 *   dalpha_qi = dout_q . v_i
 *   ds_qi     = alpha_qi (dalpha_qi - sum_j alpha_qj dalpha_qj)      (softmax)
 *   dv_i     += sum_q alpha_qi dout_q                               (value path)
 *   dk_i      = sum_q ds_qi w_q;   dw_q += sum_i ds_qi k_i
 *   dg[c]    += sum_i dk_i[c] v_i[c] / r_i
 *   dv_i[c]  += g[c] dk_i[c] / r_i - v_i[c] (sum_c' g[c'] dk_i[c'] v_i[c']) / (d r_i^3)
 * (the last line is the derivative of g * v / r; a zero source with eps = 0
 * has k = 0 and passes nothing back through its score).
 * src, dsrc [n_src][T][d]; queries, dq [n_q][d]; dout [n_q][T][d]; dg [d]
 * (the gain's gradient even when gain is NULL, i.e. 1); dq and dg are sums
 * over the tokens.
 * dlse [n_q][T] (may be NULL): the gradient of each query's log-sum-exp,
 * lse_q = log sum_i exp(s_qi) (the phase-1 state of [Summary §3 Inference]);
 * d lse_q / d s_qi = alpha_qi, so it adds alpha_qi dlse_q to ds_qi. */
int oracle_read_bwd_lse(const double *src, int64_t n_src, int64_t T, int64_t d,
                        const double *queries, int64_t n_q, const double *gain, double eps,
                        const double *dout, const double *dlse, double *dsrc, double *dq, double *dg)
{
    if (!src || !queries || !dout || !dsrc || !dq || !dg || n_src < 1 || n_q < 1 || T < 0 || d < 1 ||
        eps < 0)
        return -1;
    double *r = (double *)malloc(sizeof(double) * (size_t)n_src);
    double *k = (double *)malloc(sizeof(double) * (size_t)(n_src * d));
    double *s = (double *)malloc(sizeof(double) * (size_t)n_src);
    double *a = (double *)malloc(sizeof(double) * (size_t)(n_q * n_src));
    double *ds = (double *)malloc(sizeof(double) * (size_t)(n_q * n_src));
    double *dk = (double *)malloc(sizeof(double) * (size_t)d);
    if (!r || !k || !s || !a || !ds || !dk) {
        free(r); free(k); free(s); free(a); free(ds); free(dk);
        return -1;
    }
    for (int64_t i = 0; i < n_src * T * d; ++i) dsrc[i] = 0.0;
    for (int64_t i = 0; i < n_q * d; ++i) dq[i] = 0.0;
    for (int64_t c = 0; c < d; ++c) dg[c] = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        /* forward: normalised keys, scores, weights */
        for (int64_t i = 0; i < n_src; ++i) {
            const double *v = src + (i * T + t) * d;
            double ms = 0.0;
            for (int64_t c = 0; c < d; ++c) ms += v[c] * v[c];
            r[i] = sqrt(ms / (double)d + eps);
            for (int64_t c = 0; c < d; ++c)
                k[i * d + c] = r[i] > 0.0 ? (gain ? gain[c] : 1.0) * v[c] / r[i] : 0.0;
        }
        for (int64_t q = 0; q < n_q; ++q) {
            for (int64_t i = 0; i < n_src; ++i) {
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += queries[q * d + c] * k[i * d + c];
                s[i] = acc;
            }
            softmax(s, n_src, a + q * n_src);
            /* softmax backward */
            const double *dh = dout + (q * T + t) * d;
            double mean = 0.0;
            for (int64_t i = 0; i < n_src; ++i) {
                const double *v = src + (i * T + t) * d;
                double dal = 0.0;
                for (int64_t c = 0; c < d; ++c) dal += dh[c] * v[c];
                ds[q * n_src + i] = dal;                     /* dalpha, for now */
                mean += a[q * n_src + i] * dal;
            }
            for (int64_t i = 0; i < n_src; ++i)
                ds[q * n_src + i] = a[q * n_src + i] * (ds[q * n_src + i] - mean + (dlse ? dlse[q * T + t] : 0.0));
            /* value path and the query's gradient */
            for (int64_t i = 0; i < n_src; ++i) {
                double *dv = dsrc + (i * T + t) * d;
                for (int64_t c = 0; c < d; ++c) {
                    dv[c] += a[q * n_src + i] * dh[c];
                    dq[q * d + c] += ds[q * n_src + i] * k[i * d + c];
                }
            }
        }
        /* score path through the normalised key of every source */
        for (int64_t i = 0; i < n_src; ++i) {
            if (r[i] <= 0.0) continue;
            const double *v = src + (i * T + t) * d;
            double *dv = dsrc + (i * T + t) * d;
            for (int64_t c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int64_t q = 0; q < n_q; ++q) acc += ds[q * n_src + i] * queries[q * d + c];
                dk[c] = acc;
            }
            double gdkv = 0.0;
            for (int64_t c = 0; c < d; ++c) gdkv += (gain ? gain[c] : 1.0) * dk[c] * v[c];
            for (int64_t c = 0; c < d; ++c) {
                const double gc = gain ? gain[c] : 1.0;
                dg[c] += dk[c] * v[c] / r[i];
                dv[c] += gc * dk[c] / r[i] - v[c] * gdkv / ((double)d * r[i] * r[i] * r[i]);
            }
        }
    }
    free(r); free(k); free(s); free(a); free(ds); free(dk);
    return 0;
}

/* The read's backward without a log-sum-exp gradient. */
int oracle_read_bwd(const double *src, int64_t n_src, int64_t T, int64_t d,
                    const double *queries, int64_t n_q, const double *gain, double eps,
                    const double *dout, double *dsrc, double *dq, double *dg)
{
    return oracle_read_bwd_lse(src, n_src, T, d, queries, n_q, gain, eps, dout, NULL, dsrc, dq, dg);
}

/* Backward of the phase-2 merge (oracle_block_phase2) for an output gradient
 * dh [T][d].  Per token, with the forward
 *   r_p = sqrt(mean(p^2) + eps),  s_p = w . (g * p) / r_p,  M = max(lse, s_p),
 *   a = e^{lse-M} / (e^{lse-M} + e^{s_p-M}),  b = 1 - a,  h = a o + b p,
 * the chain rule gives
 *   d_o          = a dh
 *   dlse         = a b (dh . (o - p))          (da/dlse = a b, dh/da = o - p)
 *   ds_p         = -dlse                       (da/ds_p = -a b)
 *   d_partial    = b dh + ds_p d s_p/d p,  d s_p/d p = g*w / r_p - p (w . (g*p)) / (d r_p^3)
 *   dquery      += ds_p g * p / r_p,  dgain += ds_p w * p / r_p.
 * A zero partial with eps = 0 has no score path (s_p = 0 and nothing passes
 * back through it).  partial == NULL (the block's first layer, out = o):
 * d_o = dh, dlse = 0, and the partial, query and gain get nothing.
 * o, partial, dh, d_o, d_partial [T][d]; lse, dlse [T]; query, dquery, dgain [d]. */
int oracle_block_phase2_bwd(const double *o, const double *lse, const double *partial,
                            int64_t T, int64_t d, const double *query, const double *gain,
                            double eps, const double *dh, double *d_o, double *dlse,
                            double *d_partial, double *dquery, double *dgain)
{
    if (!o || !lse || !query || !dh || !d_o || !dlse || !dquery || !dgain || T < 0 || d < 1 || eps < 0)
        return -1;
    if (partial && !d_partial) return -1;
    for (int64_t c = 0; c < d; ++c) { dquery[c] = 0.0; dgain[c] = 0.0; }
    for (int64_t t = 0; t < T; ++t) {
        const double *ot = o + t * d, *ht = dh + t * d;
        if (!partial) {
            for (int64_t c = 0; c < d; ++c) d_o[t * d + c] = ht[c];
            dlse[t] = 0.0;
            continue;
        }
        const double *pt = partial + t * d;
        double ms = 0.0, wgp = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            ms += pt[c] * pt[c];
            wgp += query[c] * (gain ? gain[c] : 1.0) * pt[c];
        }
        const double r = sqrt(ms / (double)d + eps);
        const double sp = r > 0.0 ? wgp / r : 0.0;
        const double M = lse[t] > sp ? lse[t] : sp;
        const double ea = exp(lse[t] - M), eb = exp(sp - M);
        const double a = ea / (ea + eb), b = eb / (ea + eb);
        double hdiff = 0.0;
        for (int64_t c = 0; c < d; ++c) hdiff += ht[c] * (ot[c] - pt[c]);
        dlse[t] = a * b * hdiff;
        const double dsp = -dlse[t];
        for (int64_t c = 0; c < d; ++c) {
            const double gc = gain ? gain[c] : 1.0;
            d_o[t * d + c] = a * ht[c];
            double dp = b * ht[c];
            if (r > 0.0) {
                dp += dsp * (gc * query[c] / r - pt[c] * wgp / ((double)d * r * r * r));
                dquery[c] += dsp * gc * pt[c] / r;
                dgain[c] += dsp * query[c] * pt[c] / r;
            }
            d_partial[t * d + c] = dp;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* MHAR                                                                    */
/* ---------------------------------------------------------------------- */

/* Multi-Head Attention Residuals, [MHAR abstract]: the routing query is
 * reshaped into H heads of d/H; each head has its own softmax over the
 * depth sources; the read is block-diagonal (head h mixes only channels of
 * its own slice).  Reading taken: the RMSNorm of the key is taken per head
 * over the head's slice with the slice of the gain.  queries[n_q][H][d/H],
 * out[n_q][T][d], lse[n_q][H][T] (may be NULL). */
int oracle_mhar(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t H,
                const double *queries, int64_t n_q, const double *gain, double eps,
                double *out, double *lse)
{
    if (!src || !queries || !out || n_src < 1 || T < 0 || d < 1 || H < 1 || d % H || n_q < 1 || eps < 0)
        return -1;
    const int64_t dh = d / H;
    const double **rows = (const double **)malloc(sizeof(double *) * (size_t)n_src);
    double *h = (double *)malloc(sizeof(double) * (size_t)dh);
    if (!rows || !h) { free(rows); free(h); return -1; }
    for (int64_t q = 0; q < n_q; ++q)
        for (int64_t hd = 0; hd < H; ++hd)
            for (int64_t t = 0; t < T; ++t) {
                for (int64_t i = 0; i < n_src; ++i) rows[i] = src + (i * T + t) * d + hd * dh;
                double l;
                if (read_one(rows, n_src, dh, queries + (q * H + hd) * dh,
                             gain ? gain + hd * dh : NULL, eps, h, NULL, &l)) {
                    free(rows); free(h); return -1;
                }
                for (int64_t c = 0; c < dh; ++c) out[(q * T + t) * d + hd * dh + c] = h[c];
                if (lse) lse[(q * H + hd) * T + t] = l;
            }
    free(rows); free(h);
    return 0;
}

/* MHAR inside the two-phase Block schedule.  Phase 1 is oracle_mhar over
 * the cached block representations (it keeps lse per head); phase 2 folds in
 * the layer's partial sum head by head, each head with its own slice of the
 * query, the gain and the RMSNorm ([MHAR abstract]: every head has its own
 * softmax over the sources, the read is block-diagonal), by the merge of
 * [Summary §3 Inference, Phase 2]:
 *   s_h = w_h . RMSNorm_h(p_h),  M = max(lse_h, s_h),
 *   out_h = (e^{lse_h - M} o_h + e^{s_h - M} p_h) / (e^{lse_h - M} + e^{s_h - M}).
 * o, partial, out [T][d]; lse [H][T]; query [H][d/H]; partial == NULL copies o. */
int oracle_mhar_phase2(const double *o, const double *lse, const double *partial,
                       int64_t T, int64_t d, int64_t H, const double *query,
                       const double *gain, double eps, double *out)
{
    if (!o || !lse || !query || !out || T < 0 || d < 1 || H < 1 || d % H || eps < 0) return -1;
    const int64_t dh = d / H;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)dh);
    if (!tmp) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t hd = 0; hd < H; ++hd) {
            const double *oh = o + t * d + hd * dh;
            double *outh = out + t * d + hd * dh;
            if (!partial) { for (int64_t c = 0; c < dh; ++c) outh[c] = oh[c]; continue; }
            const double *ph = partial + t * d + hd * dh;
            const double l = lse[hd * T + t];
            double sp = score(query + hd * dh, ph, gain ? gain + hd * dh : NULL, dh, eps, tmp);
            double M = l > sp ? l : sp;
            double a = exp(l - M), b = exp(sp - M);
            for (int64_t c = 0; c < dh; ++c) outh[c] = (a * oh[c] + b * ph[c]) / (a + b);
        }
    free(tmp);
    return 0;
}

/* Backward of oracle_mhar.  [MHAR abstract]: each head is its own read over
 * its slice of the channels (the read is block-diagonal), so the gradient of
 * head h depends only on that slice of the sources, of the output gradient,
 * of the query and of the gain.  Every head's slice is gathered into
 * contiguous arrays, differentiated by oracle_read_bwd with d/H channels, and
 * the gradients are scattered back into their slices.
 * src[n_src][T][d], queries[n_q][H][d/H], dout[n_q][T][d]; outputs
 * dsrc[n_src][T][d], dq[n_q][H][d/H], dg[d]. */
int oracle_mhar_bwd(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t H,
                    const double *queries, int64_t n_q, const double *gain, double eps,
                    const double *dout, double *dsrc, double *dq, double *dg)
{
    if (!src || !queries || !dout || !dsrc || !dq || !dg || n_src < 1 || n_q < 1 || T < 0 || d < 1 ||
        H < 1 || d % H || eps < 0)
        return -1;
    const int64_t dh = d / H;
    double *s_h = (double *)malloc(sizeof(double) * (size_t)(n_src * T * dh + 1));
    double *w_h = (double *)malloc(sizeof(double) * (size_t)(n_q * dh));
    double *g_h = (double *)malloc(sizeof(double) * (size_t)dh);
    double *do_h = (double *)malloc(sizeof(double) * (size_t)(n_q * T * dh + 1));
    double *ds_h = (double *)malloc(sizeof(double) * (size_t)(n_src * T * dh + 1));
    double *dq_h = (double *)malloc(sizeof(double) * (size_t)(n_q * dh));
    double *dg_h = (double *)malloc(sizeof(double) * (size_t)dh);
    int rc = (s_h && w_h && g_h && do_h && ds_h && dq_h && dg_h) ? 0 : -1;
    for (int64_t hd = 0; hd < H && rc == 0; ++hd) {
        const int64_t c0 = hd * dh;
        for (int64_t i = 0; i < n_src; ++i)
            for (int64_t t = 0; t < T; ++t)
                for (int64_t c = 0; c < dh; ++c) s_h[(i * T + t) * dh + c] = src[(i * T + t) * d + c0 + c];
        for (int64_t q = 0; q < n_q; ++q) {
            for (int64_t c = 0; c < dh; ++c) w_h[q * dh + c] = queries[q * d + c0 + c];
            for (int64_t t = 0; t < T; ++t)
                for (int64_t c = 0; c < dh; ++c) do_h[(q * T + t) * dh + c] = dout[(q * T + t) * d + c0 + c];
        }
        for (int64_t c = 0; c < dh; ++c) g_h[c] = gain ? gain[c0 + c] : 1.0;
        rc = oracle_read_bwd(s_h, n_src, T, dh, w_h, n_q, g_h, eps, do_h, ds_h, dq_h, dg_h);
        if (rc) break;
        for (int64_t i = 0; i < n_src; ++i)
            for (int64_t t = 0; t < T; ++t)
                for (int64_t c = 0; c < dh; ++c) dsrc[(i * T + t) * d + c0 + c] = ds_h[(i * T + t) * dh + c];
        for (int64_t q = 0; q < n_q; ++q)
            for (int64_t c = 0; c < dh; ++c) dq[q * d + c0 + c] = dq_h[q * dh + c];
        for (int64_t c = 0; c < dh; ++c) dg[c0 + c] = dg_h[c];
    }
    free(s_h); free(w_h); free(g_h); free(do_h); free(ds_h); free(dq_h); free(dg_h);
    return rc;
}

/* ---------------------------------------------------------------------- */
/* MSAR                                                                    */
/* ---------------------------------------------------------------------- */

/* Stream expansion, [MSAR §무엇과 다른가]: stream 0 is the identity; stream
 * r >= 1 is a causal depthwise 1-D convolution along the token axis with
 * kernel size k_r.  Readings taken: left zero padding, no bias,
 *   u^(r)[t][c] = sum_{j<k_r} cw_r[c][j] * v[t-j][c]   (v[t<0] = 0).
 * conv_w packs the m-1 kernels one after the other, kernel r as [d][k_r].
 * v[T][d] (one source), u[T][d]. */
int oracle_msar_conv(const double *v, int64_t T, int64_t d, int64_t k,
                     const double *cw, double *u)
{
    if (!v || !cw || !u || T < 0 || d < 1 || k < 1) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < k; ++j)
                if (t - j >= 0) acc += cw[c * k + j] * v[(t - j) * d + c];
            u[t * d + c] = acc;
        }
    return 0;
}

/* H^pre mixer of one token, [MSAR §무엇과 다른가]: z = RMSNorm(Flatten(Z))
 * over m*d (stream-major: element r*d + c is Z^(r)[c]); c = sigmoid(z^T P)
 * with P [m*d][m]; h = sum_r c_r Z^(r).  Z[m][d] -> out[d]; zf[m*d] and
 * logit[m] are scratch; mixc (may be NULL) receives c. */
static void msar_mix(const double *Z, int64_t m, int64_t d, const double *mix_gain,
                     const double *mix_w, double mix_eps, double *zf, double *logit,
                     double *out, double *mixc)
{
    rmsnorm(Z, mix_gain, m * d, mix_eps, zf);
    for (int64_t o = 0; o < m; ++o) {
        double acc = 0.0;
        for (int64_t k = 0; k < m * d; ++k) acc += zf[k] * mix_w[k * m + o];
        logit[o] = 1.0 / (1.0 + exp(-acc));
        if (mixc) mixc[o] = logit[o];
    }
    for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t r = 0; r < m; ++r) acc += logit[r] * Z[r * d + c];
        out[c] = acc;
    }
}

/* The m streams of one source, [MSAR §무엇과 다른가]: u[r][T][d] with u[0] = v
 * and u[r] the causal conv of v with kernel r (conv_w packed as above). */
static int msar_expand(const double *v, int64_t T, int64_t d, int64_t m, const int32_t *ksizes,
                       const double *conv_w, double *u)
{
    size_t per = (size_t)T * (size_t)d;
    int64_t off = 0;
    for (int64_t r = 0; r < m; ++r) {
        double *ur = u + (size_t)r * per;
        if (r == 0) memcpy(ur, v, sizeof(double) * per);
        else {
            if (oracle_msar_conv(v, T, d, ksizes[r - 1], conv_w + off, ur)) return -1;
            off += d * (int64_t)ksizes[r - 1];
        }
    }
    return 0;
}

/* MSAR read for one target layer, [MSAR §무엇과 다른가]:
 *   1. every source v_i is expanded into m full-width streams u_i^(r);
 *   2. each stream r reads the depth history with its own pseudo-query
 *      w^(r): Z^(r) = sum_i softmax_i(w^(r)T RMSNorm(u_i^(r))) u_i^(r)
 *      (each stream's weights sum to 1);
 *   3. H^pre mixer: z = RMSNorm(Flatten(Z)) over m*d (flattened stream-major,
 *      element r*d + c is Z^(r)[c]); c = sigmoid(z^T P) with P [m*d][m];
 *      h = sum_r c_r Z^(r).
 * Readings taken: plain sigmoid, weights not renormalised, no bias.
 * src[n_src][T][d]; ksizes[m-1]; conv_w packed; queries[m][d]; gain[d] or
 * NULL; mix_gain[m*d] or NULL; mix_w[m*d][m]; out[T][d].
 * Optional debug outputs (may be NULL): alpha[T][m][n_src], mixc[T][m]. */
int oracle_msar(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t m,
                const int32_t *ksizes, const double *conv_w, const double *queries,
                const double *gain, double eps, const double *mix_gain,
                const double *mix_w, double mix_eps, double *out,
                double *alpha, double *mixc)
{
    if (!src || !ksizes || !conv_w || !queries || !mix_w || !out || n_src < 1 || T < 0 ||
        d < 1 || m < 1 || eps < 0 || mix_eps < 0) return -1;
    /* expanded streams u[r][i][T][d] */
    size_t per = (size_t)T * (size_t)d;
    double *u = (double *)malloc(sizeof(double) * (size_t)m * (size_t)n_src * per + 1);
    double *Z = (double *)malloc(sizeof(double) * (size_t)m * (size_t)d + 1);
    double *zf = (double *)malloc(sizeof(double) * (size_t)m * (size_t)d + 1);
    const double **rows = (const double **)malloc(sizeof(double *) * (size_t)n_src);
    double *a = (double *)malloc(sizeof(double) * (size_t)n_src);
    double *logit = (double *)malloc(sizeof(double) * (size_t)m);
    if (!u || !Z || !zf || !rows || !a || !logit) goto fail;
    {
        int64_t off = 0;
        for (int64_t r = 0; r < m; ++r) {
            for (int64_t i = 0; i < n_src; ++i) {
                const double *v = src + (size_t)i * per;
                double *ur = u + ((size_t)r * (size_t)n_src + (size_t)i) * per;
                if (r == 0) memcpy(ur, v, sizeof(double) * per);
                else if (oracle_msar_conv(v, T, d, ksizes[r - 1], conv_w + off, ur)) goto fail;
            }
            if (r >= 1) off += d * (int64_t)ksizes[r - 1];
        }
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t r = 0; r < m; ++r) {
                for (int64_t i = 0; i < n_src; ++i)
                    rows[i] = u + ((size_t)r * (size_t)n_src + (size_t)i) * per + (size_t)t * (size_t)d;
                if (read_one(rows, n_src, d, queries + r * d, gain, eps, Z + r * d, a, NULL)) goto fail;
                if (alpha) for (int64_t i = 0; i < n_src; ++i) alpha[(t * m + r) * n_src + i] = a[i];
            }
            msar_mix(Z, m, d, mix_gain, mix_w, mix_eps, zf, logit, out + t * d, mixc ? mixc + t * m : NULL);
        }
    }
    free(u); free(Z); free(zf); free(rows); free(a); free(logit);
    return 0;
fail:
    free(u); free(Z); free(zf); free(rows); free(a); free(logit);
    return -1;
}

/* MSAR read with each source's own conv kernels: source i is expanded with
 * the kernels packed at conv_w + i * conv_src_stride (as oracle_msar's
 * conv_w for that source; the streams of a source are the source's own,
 * [MSAR §무엇과 다른가] v_i^(r)); the per-stream reads and the mixer are
 * oracle_msar's.  conv_src_stride = 0 is oracle_msar. */
int oracle_msar_ps(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t m,
                   const int32_t *ksizes, const double *conv_w, int64_t conv_src_stride,
                   const double *queries, const double *gain, double eps, const double *mix_gain,
                   const double *mix_w, double mix_eps, double *out)
{
    if (!src || !ksizes || !conv_w || !queries || !mix_w || !out || n_src < 1 || T < 0 || d < 1 ||
        m < 1 || eps < 0 || mix_eps < 0 || conv_src_stride < 0) return -1;
    size_t per = (size_t)T * (size_t)d;
    /* u[i][r][T][d] */
    double *u = (double *)malloc(sizeof(double) * (size_t)n_src * (size_t)m * per + 1);
    double *Z = (double *)malloc(sizeof(double) * (size_t)m * (size_t)d + 1);
    double *zf = (double *)malloc(sizeof(double) * (size_t)m * (size_t)d + 1);
    double *logit = (double *)malloc(sizeof(double) * (size_t)m);
    const double **rows = (const double **)malloc(sizeof(double *) * (size_t)n_src);
    int rc = (u && Z && zf && logit && rows) ? 0 : -1;
    for (int64_t i = 0; i < n_src && rc == 0; ++i)
        rc = msar_expand(src + (size_t)i * per, T, d, m, ksizes, conv_w + i * conv_src_stride,
                         u + (size_t)i * (size_t)m * per);
    for (int64_t t = 0; t < T && rc == 0; ++t) {
        for (int64_t r = 0; r < m && rc == 0; ++r) {
            for (int64_t i = 0; i < n_src; ++i)
                rows[i] = u + ((size_t)i * (size_t)m + (size_t)r) * per + (size_t)t * (size_t)d;
            rc = read_one(rows, n_src, d, queries + r * d, gain, eps, Z + r * d, NULL, NULL);
        }
        if (rc == 0) msar_mix(Z, m, d, mix_gain, mix_w, mix_eps, zf, logit, out + t * d, NULL);
    }
    free(u); free(Z); free(zf); free(logit); free(rows);
    return rc;
}

/* Backward of the H^pre mixer (msar_mix) for one token, [MSAR 무엇과 다른가]:
 *   dc_r   = dh . Z^(r);  dl_o = dc_o c_o (1 - c_o)     (c = sigmoid(l))
 *   dzn    = sum_o dl_o P[:, o];  dP[:, o] += dl_o zn;  dmix_gain += dzn * zf / nu
 *   dzf    = mg * dzn / nu - zf (sum_k mg_k dzn_k zf_k) / (m d nu^3)   (RMSNorm over m d)
 *   dZ^(r) = c_r dh + dzf[r d .. (r+1) d)
 * Z^(r) of the token at Zt + r * zstride, dZ^(r) written at dZt + r * dzstride;
 * dmix_gain and dmix_w are added into; zf, zn, dzn [m d] and c, dl [m] are
 * scratch. */
static void msar_mix_bwd_token(const double *Zt, size_t zstride, const double *ht, int64_t m, int64_t d,
                               const double *mix_gain, const double *mix_w, double mix_eps, double *zf, double *zn,
                               double *dzn, double *c, double *dl, double *dZt, size_t dzstride, double *dmix_gain,
                               double *dmix_w)
{
    const size_t md = (size_t)m * (size_t)d;
    for (int64_t r = 0; r < m; ++r)
        for (int64_t k = 0; k < d; ++k) zf[r * d + k] = Zt[(size_t)r * zstride + (size_t)k];
    double ms = 0.0;
    for (size_t k = 0; k < md; ++k) ms += zf[k] * zf[k];
    const double nu = sqrt(ms / (double)md + mix_eps);
    for (size_t k = 0; k < md; ++k) zn[k] = nu > 0.0 ? (mix_gain ? mix_gain[k] : 1.0) * zf[k] / nu : 0.0;
    for (int64_t o = 0; o < m; ++o) {
        double acc = 0.0;
        for (size_t k = 0; k < md; ++k) acc += zn[k] * mix_w[k * m + o];
        c[o] = 1.0 / (1.0 + exp(-acc));
        double dc = 0.0;
        for (int64_t k = 0; k < d; ++k) dc += ht[k] * zf[o * d + k];
        dl[o] = dc * c[o] * (1.0 - c[o]);
    }
    double s = 0.0;
    for (size_t k = 0; k < md; ++k) {
        double acc = 0.0;
        for (int64_t o = 0; o < m; ++o) {
            acc += dl[o] * mix_w[k * m + o];
            dmix_w[k * m + o] += dl[o] * zn[k];
        }
        dzn[k] = acc;
        if (nu > 0.0) dmix_gain[k] += acc * zf[k] / nu;
        s += (mix_gain ? mix_gain[k] : 1.0) * acc * zf[k];
    }
    for (int64_t r = 0; r < m; ++r)
        for (int64_t k = 0; k < d; ++k) {
            const size_t kk = (size_t)r * (size_t)d + (size_t)k;
            double dzf = 0.0;
            if (nu > 0.0)
                dzf = (mix_gain ? mix_gain[kk] : 1.0) * dzn[kk] / nu - zf[kk] * s / ((double)md * nu * nu * nu);
            dZt[(size_t)r * dzstride + (size_t)k] = c[r] * ht[k] + dzf;
        }
}

/* Transpose of one causal depthwise conv (oracle_msar_conv) of source v with
 * kernel cw [d][kr]: for u[t][c] = sum_j cw[c][j] v[t-j][c] and its gradient
 * dui, dv[t-j][c] += cw[c][j] dui[t][c] and dcw[c][j] += dui[t][c] v[t-j][c]
 * (both added into). */
static void conv_transpose(const double *v, const double *dui, int64_t T, int64_t d, int64_t kr,
                           const double *cw, double *dv, double *dcw)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < d; ++k)
            for (int64_t j = 0; j < kr; ++j)
                if (t - j >= 0) {
                    dv[(t - j) * d + k] += cw[k * kr + j] * dui[t * d + k];
                    dcw[k * kr + j] += dui[t * d + k] * v[(t - j) * d + k];
                }
}

/* Backward of the MSAR read (oracle_msar) for an output gradient dh[T][d].
 * The forward is taken apart as in oracle_msar: streams u_i^(r), per-stream
 * reads Z^(r) (read_one), and the H^pre mixer.  Chain rule, per token:
 *   mixer   dc_r   = dh . Z^(r);  dl_o = dc_o c_o (1 - c_o)     (c = sigmoid(l))
 *           dzn    = sum_o dl_o P[:, o];  dP[:, o] += dl_o zn;  dmix_gain += dzn * zf / nu
 *           dzf    = mg * dzn / nu - zf (sum_k mg_k dzn_k zf_k) / (m d nu^3)   (RMSNorm over m d)
 *           dZ^(r) = c_r dh + dzf[r d .. (r+1) d)
 *   reads   each stream r is a read of the sources u_i^(r) with query w_r:
 *           oracle_read_bwd gives du_i^(r), dw_r and stream r's share of dgain
 *   streams dv_i[t] += du_i^(0)[t];  for r >= 1, u^(r)[t][c] = sum_j cw_r[c][j] v[t-j][c]:
 *           dv_i[t-j][c] += cw_r[c][j] du_i^(r)[t][c],  dcw_r[c][j] += du_i^(r)[t][c] v_i[t-j][c]
 * Outputs: dsrc[n_src][T][d], dconv_w (packed as conv_w), dq[m][d], dg[d],
 * dmix_gain[m*d], dmix_w[m*d][m]. */
/* Shared by the two entry points below: conv_src_stride = 0 gives every
 * source the kernels at conv_w and sums dconv_w over the sources; > 0 gives
 * source i the kernels at conv_w + i * conv_src_stride and its own gradient at
 * dconv_w + i * conv_src_stride (the per-source reading of oracle_msar_ps). */
static int msar_bwd_impl(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t m,
                         const int32_t *ksizes, const double *conv_w, int64_t conv_src_stride,
                         const double *queries, const double *gain, double eps, const double *mix_gain,
                         const double *mix_w, double mix_eps, const double *dh, double *dsrc, double *dconv_w,
                         double *dq, double *dg, double *dmix_gain, double *dmix_w)
{
    if (!src || !ksizes || !conv_w || !queries || !mix_w || !dh || !dsrc || !dconv_w || !dq || !dg ||
        !dmix_gain || !dmix_w || n_src < 1 || T < 0 || d < 1 || m < 1 || eps < 0 || mix_eps < 0 ||
        conv_src_stride < 0)
        return -1;
    const size_t per = (size_t)T * (size_t)d, md = (size_t)m * (size_t)d;
    int64_t ktot = 0;
    for (int64_t r = 0; r + 1 < m; ++r) ktot += ksizes[r];
    double *u = (double *)malloc(sizeof(double) * (size_t)m * (size_t)n_src * per + 1);    /* [r][i][T][d] */
    double *Z = (double *)malloc(sizeof(double) * md * (size_t)T + 1);                     /* [r][T][d] */
    double *dZ = (double *)malloc(sizeof(double) * md * (size_t)T + 1);                    /* [r][T][d] */
    double *du = (double *)malloc(sizeof(double) * (size_t)n_src * per + 1);               /* [i][T][d] */
    double *dqr = (double *)malloc(sizeof(double) * (size_t)d);
    double *dgr = (double *)malloc(sizeof(double) * (size_t)d);
    double *zf = (double *)malloc(sizeof(double) * md + 1);
    double *zn = (double *)malloc(sizeof(double) * md + 1);
    double *dzn = (double *)malloc(sizeof(double) * md + 1);
    double *c = (double *)malloc(sizeof(double) * (size_t)m);
    double *dl = (double *)malloc(sizeof(double) * (size_t)m);
    const double **rows = (const double **)malloc(sizeof(double *) * (size_t)n_src);
    int rc = (u && Z && dZ && du && dqr && dgr && zf && zn && dzn && c && dl && rows) ? 0 : -1;
    for (size_t k = 0; rc == 0 && k < (size_t)n_src * per; ++k) dsrc[k] = 0.0;
    for (int64_t i = 0; rc == 0 && i < (conv_src_stride ? n_src : 1); ++i)
        for (int64_t k = 0; k < d * ktot; ++k) dconv_w[i * conv_src_stride + k] = 0.0;
    for (size_t k = 0; rc == 0 && k < md; ++k) { dmix_gain[k] = 0.0; for (int64_t o = 0; o < m; ++o) dmix_w[k * m + o] = 0.0; }
    for (int64_t k = 0; rc == 0 && k < d; ++k) dg[k] = 0.0;
    /* forward: streams and per-stream reads */
    for (int64_t r = 0, off = 0; r < m && rc == 0; ++r) {
        for (int64_t i = 0; i < n_src && rc == 0; ++i) {
            const double *v = src + (size_t)i * per;
            double *ur = u + ((size_t)r * (size_t)n_src + (size_t)i) * per;
            if (r == 0) memcpy(ur, v, sizeof(double) * per);
            else rc = oracle_msar_conv(v, T, d, ksizes[r - 1], conv_w + i * conv_src_stride + off, ur);
        }
        if (r >= 1) off += d * (int64_t)ksizes[r - 1];
        for (int64_t t = 0; t < T && rc == 0; ++t) {
            for (int64_t i = 0; i < n_src; ++i) rows[i] = u + ((size_t)r * (size_t)n_src + (size_t)i) * per + (size_t)t * (size_t)d;
            rc = read_one(rows, n_src, d, queries + r * d, gain, eps, Z + (size_t)r * per + (size_t)t * (size_t)d, NULL, NULL);
        }
    }
    /* mixer backward, per token */
    for (int64_t t = 0; t < T && rc == 0; ++t)
        msar_mix_bwd_token(Z + (size_t)t * (size_t)d, per, dh + t * d, m, d, mix_gain, mix_w, mix_eps, zf, zn, dzn,
                           c, dl, dZ + (size_t)t * (size_t)d, per, dmix_gain, dmix_w);
    /* per-stream read backward, then back through the streams */
    for (int64_t r = 0, off = 0; r < m && rc == 0; ++r) {
        rc = oracle_read_bwd(u + (size_t)r * (size_t)n_src * per, n_src, T, d, queries + r * d, 1, gain, eps,
                             dZ + (size_t)r * per, du, dqr, dgr);
        if (rc) break;
        for (int64_t k = 0; k < d; ++k) { dq[r * d + k] = dqr[k]; dg[k] += dgr[k]; }
        if (r == 0) {
            for (size_t k = 0; k < (size_t)n_src * per; ++k) dsrc[k] += du[k];
            continue;
        }
        const int64_t kr = ksizes[r - 1];
        for (int64_t i = 0; i < n_src; ++i) {
            const double *cw = conv_w + i * conv_src_stride + off;
            double *dcw = dconv_w + i * conv_src_stride + off;
            conv_transpose(src + (size_t)i * per, du + (size_t)i * per, T, d, kr, cw, dsrc + (size_t)i * per, dcw);
        }
        off += d * kr;
    }
    free(u); free(Z); free(dZ); free(du); free(dqr); free(dgr); free(zf); free(zn); free(dzn); free(c); free(dl);
    free(rows);
    return rc;
}

int oracle_msar_bwd(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t m,
                    const int32_t *ksizes, const double *conv_w, const double *queries,
                    const double *gain, double eps, const double *mix_gain, const double *mix_w,
                    double mix_eps, const double *dh, double *dsrc, double *dconv_w, double *dq,
                    double *dg, double *dmix_gain, double *dmix_w)
{
    return msar_bwd_impl(src, n_src, T, d, m, ksizes, conv_w, 0, queries, gain, eps, mix_gain, mix_w, mix_eps,
                         dh, dsrc, dconv_w, dq, dg, dmix_gain, dmix_w);
}

/* Backward of oracle_msar_ps (each source's own kernels, conv_src_stride > 0
 * floats apart): the chain rule of oracle_msar_bwd with source i's streams
 * taken through its own kernels, and dconv_w written per source at the same
 * stride (the floats between one source's kernels and the next are left
 * untouched).  [MSAR 무엇과 다른가], the streams v_i^(r) of each source. */
int oracle_msar_ps_bwd(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t m,
                       const int32_t *ksizes, const double *conv_w, int64_t conv_src_stride,
                       const double *queries, const double *gain, double eps, const double *mix_gain,
                       const double *mix_w, double mix_eps, const double *dh, double *dsrc, double *dconv_w,
                       double *dq, double *dg, double *dmix_gain, double *dmix_w)
{
    if (conv_src_stride < 1) return -1;
    return msar_bwd_impl(src, n_src, T, d, m, ksizes, conv_w, conv_src_stride, queries, gain, eps, mix_gain,
                         mix_w, mix_eps, dh, dsrc, dconv_w, dq, dg, dmix_gain, dmix_w);
}

/* MSAR inside the two-phase Block schedule, phase 1.  [MSAR §어떻게 쓰나]:
 * AttnRes's two-phase computation carries over to MSAR unchanged: every
 * target query of the block is read against the completed sources in one
 * batch, and each layer later merges its own partial-sum contribution by the
 * online softmax.  Reading taken: the streams of a source belong to the
 * source (the page writes them v_i^(r), with no layer index), so one set of
 * conv kernels serves every layer of the block and each cached source is
 * expanded once.  For every layer s and stream r this keeps the read's state
 * over the cached sources, as phase 1 of [Summary §3 Inference]:
 *   o_s^(r)   = sum_i softmax_i(w_s^(r)T RMSNorm(u_i^(r))) u_i^(r)
 *   lse_s^(r) = log sum_i exp(w_s^(r)T RMSNorm(u_i^(r))).
 * src[n_src][T][d]; queries[S][m][d]; o[S][m][T][d]; lse[S][m][T]. */
int oracle_msar_phase1(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t m,
                       const int32_t *ksizes, const double *conv_w, const double *queries,
                       int64_t S, const double *gain, double eps, double *o, double *lse)
{
    if (!src || !ksizes || !conv_w || !queries || !o || !lse || n_src < 1 || T < 0 || d < 1 ||
        m < 1 || S < 1 || eps < 0) return -1;
    size_t per = (size_t)T * (size_t)d;
    /* u[i][r][T][d]: the streams of every source, expanded once */
    double *u = (double *)malloc(sizeof(double) * (size_t)n_src * (size_t)m * per + 1);
    const double **rows = (const double **)malloc(sizeof(double *) * (size_t)n_src);
    int rc = (u && rows) ? 0 : -1;
    for (int64_t i = 0; i < n_src && rc == 0; ++i)
        rc = msar_expand(src + (size_t)i * per, T, d, m, ksizes, conv_w, u + (size_t)i * (size_t)m * per);
    for (int64_t sl = 0; sl < S && rc == 0; ++sl)
        for (int64_t r = 0; r < m && rc == 0; ++r)
            for (int64_t t = 0; t < T && rc == 0; ++t) {
                for (int64_t i = 0; i < n_src; ++i)
                    rows[i] = u + ((size_t)i * (size_t)m + (size_t)r) * per + (size_t)t * (size_t)d;
                rc = read_one(rows, n_src, d, queries + (sl * m + r) * d, gain, eps,
                              o + (((size_t)sl * (size_t)m + (size_t)r) * (size_t)T + (size_t)t) * (size_t)d,
                              NULL, lse + (sl * m + r) * T + t);
            }
    free(u); free(rows);
    return rc;
}

/* MSAR two-phase, phase 2 for one layer.  The layer's partial sum p is its
 * one more source ([Summary §2 Block AttnRes]); it is expanded into m streams
 * with the same kernels, causally over p's own history ([MSAR §무엇과 다른가]).
 * Each stream's score s_p^(r) = w^(r)T RMSNorm(u_p^(r)) is merged into that
 * stream's phase-1 state by the merge of [Summary §3 Inference, Phase 2]:
 *   M = max(lse^(r), s_p^(r)),
 *   Z^(r) = (e^{lse^(r)-M} o^(r) + e^{s_p^(r)-M} u_p^(r)) / (e^{lse^(r)-M} + e^{s_p^(r)-M}),
 * and the merged states go through the H^pre mixer (msar_mix).  partial ==
 * NULL (the block's first layer) takes Z^(r) = o^(r).
 * o[m][T][d]; lse[m][T]; partial[T][d] or NULL; query[m][d]; out[T][d]. */
int oracle_msar_phase2(const double *o, const double *lse, const double *partial, int64_t T,
                       int64_t d, int64_t m, const int32_t *ksizes, const double *conv_w,
                       const double *query, const double *gain, double eps,
                       const double *mix_gain, const double *mix_w, double mix_eps, double *out)
{
    if (!o || !lse || !ksizes || !conv_w || !query || !mix_w || !out || T < 0 || d < 1 || m < 1 ||
        eps < 0 || mix_eps < 0) return -1;
    size_t per = (size_t)T * (size_t)d;
    double *up = partial ? (double *)malloc(sizeof(double) * (size_t)m * per + 1) : NULL;
    double *Z = (double *)malloc(sizeof(double) * (size_t)m * (size_t)d + 1);
    double *zf = (double *)malloc(sizeof(double) * (size_t)m * (size_t)d + 1);
    double *logit = (double *)malloc(sizeof(double) * (size_t)m);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = (Z && zf && logit && tmp && (!partial || up)) ? 0 : -1;
    if (rc == 0 && partial) rc = msar_expand(partial, T, d, m, ksizes, conv_w, up);
    for (int64_t t = 0; t < T && rc == 0; ++t) {
        for (int64_t r = 0; r < m; ++r) {
            const double *orow = o + ((size_t)r * (size_t)T + (size_t)t) * (size_t)d;
            double *zr = Z + r * d;
            if (!partial) { for (int64_t c = 0; c < d; ++c) zr[c] = orow[c]; continue; }
            const double *prow = up + (size_t)r * per + (size_t)t * (size_t)d;
            const double l = lse[r * T + t];
            double sp = score(query + r * d, prow, gain, d, eps, tmp);
            double M = l > sp ? l : sp;
            double a = exp(l - M), b = exp(sp - M);
            for (int64_t c = 0; c < d; ++c) zr[c] = (a * orow[c] + b * prow[c]) / (a + b);
        }
        msar_mix(Z, m, d, mix_gain, mix_w, mix_eps, zf, logit, out + t * d, NULL);
    }
    free(up); free(Z); free(zf); free(logit); free(tmp);
    return rc;
}


/* Backward of MSAR phase 2 for one layer (oracle_msar_phase2) for an output
 * gradient dh[T][d], by the chain rule through its three steps: the partial's
 * streams (msar_expand), each stream's merge into its phase-1 state
 * ([Summary §3 Inference, Phase 2]; backward as oracle_block_phase2_bwd, the
 * stream being the merge's partial and w^(r) its query), and the H^pre mixer
 * over the merged states (msar_mix_bwd_token).  The partial's streams go back
 * through the causal convolutions (conv_transpose).
 * Outputs: d_o[m][T][d], d_lse[m][T], d_partial[T][d] (when partial != NULL),
 * dconv_w (packed as conv_w; the partial's share, zero without a partial),
 * dquery[m][d] and dgain[d] (the merges' shares), dmix_gain[m*d],
 * dmix_w[m*d][m].  partial == NULL: Z^(r) = o^(r), so d_o = dZ and
 * d_lse = 0. */
int oracle_msar_phase2_bwd(const double *o, const double *lse, const double *partial, int64_t T, int64_t d,
                           int64_t m, const int32_t *ksizes, const double *conv_w, const double *query,
                           const double *gain, double eps, const double *mix_gain, const double *mix_w,
                           double mix_eps, const double *dh, double *d_o, double *d_lse, double *d_partial,
                           double *dconv_w, double *dquery, double *dgain, double *dmix_gain, double *dmix_w)
{
    if (!o || !lse || !ksizes || !conv_w || !query || !mix_w || !dh || !d_o || !d_lse || !dconv_w || !dquery ||
        !dgain || !dmix_gain || !dmix_w || T < 0 || d < 1 || m < 1 || eps < 0 || mix_eps < 0)
        return -1;
    if (partial && !d_partial) return -1;
    const size_t per = (size_t)T * (size_t)d, md = (size_t)m * (size_t)d;
    int64_t ktot = 0;
    for (int64_t r = 0; r + 1 < m; ++r) ktot += ksizes[r];
    double *up = partial ? (double *)malloc(sizeof(double) * (size_t)m * per + 1) : NULL;     /* [r][T][d] */
    double *Z = (double *)malloc(sizeof(double) * md * (size_t)T + 1);                       /* [r][T][d] */
    double *dZ = (double *)malloc(sizeof(double) * md * (size_t)T + 1);
    double *dup = (double *)malloc(sizeof(double) * per + 1);
    double *dqr = (double *)malloc(sizeof(double) * (size_t)d);
    double *dgr = (double *)malloc(sizeof(double) * (size_t)d);
    double *zf = (double *)malloc(sizeof(double) * md + 1);
    double *zn = (double *)malloc(sizeof(double) * md + 1);
    double *dzn = (double *)malloc(sizeof(double) * md + 1);
    double *c = (double *)malloc(sizeof(double) * (size_t)m);
    double *dl = (double *)malloc(sizeof(double) * (size_t)m);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = (Z && dZ && dup && dqr && dgr && zf && zn && dzn && c && dl && tmp && (!partial || up)) ? 0 : -1;
    for (int64_t k = 0; rc == 0 && k < d * ktot; ++k) dconv_w[k] = 0.0;
    for (size_t k = 0; rc == 0 && k < md; ++k) {
        dquery[k] = 0.0;
        dmix_gain[k] = 0.0;
        for (int64_t q = 0; q < m; ++q) dmix_w[k * m + q] = 0.0;
    }
    for (int64_t k = 0; rc == 0 && k < d; ++k) dgain[k] = 0.0;
    for (size_t k = 0; rc == 0 && partial && k < per; ++k) d_partial[k] = 0.0;
    /* forward: the partial's streams and the merged states */
    if (partial && rc == 0) rc = msar_expand(partial, T, d, m, ksizes, conv_w, up);
    for (int64_t r = 0; r < m && rc == 0; ++r)
        for (int64_t t = 0; t < T; ++t) {
            const double *orow = o + (size_t)r * per + (size_t)t * (size_t)d;
            double *zr = Z + (size_t)r * per + (size_t)t * (size_t)d;
            if (!partial) { for (int64_t k = 0; k < d; ++k) zr[k] = orow[k]; continue; }
            const double *prow = up + (size_t)r * per + (size_t)t * (size_t)d;
            const double l = lse[r * T + t];
            const double sp = score(query + r * d, prow, gain, d, eps, tmp);
            const double M = l > sp ? l : sp;
            const double a = exp(l - M), b = exp(sp - M);
            for (int64_t k = 0; k < d; ++k) zr[k] = (a * orow[k] + b * prow[k]) / (a + b);
        }
    /* mixer backward, per token */
    for (int64_t t = 0; t < T && rc == 0; ++t)
        msar_mix_bwd_token(Z + (size_t)t * (size_t)d, per, dh + t * d, m, d, mix_gain, mix_w, mix_eps, zf, zn, dzn,
                           c, dl, dZ + (size_t)t * (size_t)d, per, dmix_gain, dmix_w);
    /* each stream's merge backward, then the partial's streams back through the convolutions */
    for (int64_t r = 0, off = 0; r < m && rc == 0; ++r) {
        rc = oracle_block_phase2_bwd(o + (size_t)r * per, lse + r * T, partial ? up + (size_t)r * per : NULL, T, d,
                                     query + r * d, gain, eps, dZ + (size_t)r * per, d_o + (size_t)r * per,
                                     d_lse + r * T, partial ? dup : NULL, dqr, dgr);
        if (rc) break;
        for (int64_t k = 0; k < d; ++k) { dquery[r * d + k] = dqr[k]; dgain[k] += dgr[k]; }
        if (!partial) continue;
        if (r == 0) {
            for (size_t k = 0; k < per; ++k) d_partial[k] += dup[k];
            continue;
        }
        const int64_t kr = ksizes[r - 1];
        conv_transpose(partial, dup, T, d, kr, conv_w + off, d_partial, dconv_w + off);
        off += d * kr;
    }
    free(up); free(Z); free(dZ); free(dup); free(dqr); free(dgr); free(zf); free(zn); free(dzn); free(c); free(dl);
    free(tmp);
    return rc;
}

/* Backward of MSAR phase 1 (oracle_msar_phase1) for gradients d_o[S][m][T][d]
 * and d_lse[S][m][T] of its state: for each stream r, the read of the cached
 * sources' streams u_i^(r) by the S layers' queries w_s^(r) is differentiated
 * with its lse (oracle_read_bwd_lse), and the streams go back through the
 * causal convolutions (conv_transpose).
 * Outputs: dsrc[n_src][T][d], dconv_w (packed as conv_w), dqueries[S][m][d],
 * dgain[d]. */
int oracle_msar_phase1_bwd(const double *src, int64_t n_src, int64_t T, int64_t d, int64_t m,
                           const int32_t *ksizes, const double *conv_w, const double *queries, int64_t S,
                           const double *gain, double eps, const double *d_o, const double *d_lse, double *dsrc,
                           double *dconv_w, double *dqueries, double *dgain)
{
    if (!src || !ksizes || !conv_w || !queries || !d_o || !d_lse || !dsrc || !dconv_w || !dqueries || !dgain ||
        n_src < 1 || T < 0 || d < 1 || m < 1 || S < 1 || eps < 0)
        return -1;
    const size_t per = (size_t)T * (size_t)d;
    int64_t ktot = 0;
    for (int64_t r = 0; r + 1 < m; ++r) ktot += ksizes[r];
    double *ue = (double *)malloc(sizeof(double) * (size_t)n_src * (size_t)m * per + 1);   /* [i][r][T][d] */
    double *ur = (double *)malloc(sizeof(double) * (size_t)n_src * per + 1);               /* [i][T][d] */
    double *du = (double *)malloc(sizeof(double) * (size_t)n_src * per + 1);
    double *qr = (double *)malloc(sizeof(double) * (size_t)S * (size_t)d);
    double *dor = (double *)malloc(sizeof(double) * (size_t)S * per + 1);
    double *dlr = (double *)malloc(sizeof(double) * (size_t)S * (size_t)T + 1);
    double *dqr = (double *)malloc(sizeof(double) * (size_t)S * (size_t)d);
    double *dgr = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = (ue && ur && du && qr && dor && dlr && dqr && dgr) ? 0 : -1;
    for (size_t k = 0; rc == 0 && k < (size_t)n_src * per; ++k) dsrc[k] = 0.0;
    for (int64_t k = 0; rc == 0 && k < d * ktot; ++k) dconv_w[k] = 0.0;
    for (int64_t k = 0; rc == 0 && k < d; ++k) dgain[k] = 0.0;
    for (int64_t i = 0; i < n_src && rc == 0; ++i)
        rc = msar_expand(src + (size_t)i * per, T, d, m, ksizes, conv_w, ue + (size_t)i * (size_t)m * per);
    for (int64_t r = 0, off = 0; r < m && rc == 0; ++r) {
        for (int64_t i = 0; i < n_src; ++i)
            memcpy(ur + (size_t)i * per, ue + ((size_t)i * (size_t)m + (size_t)r) * per, sizeof(double) * per);
        for (int64_t sl = 0; sl < S; ++sl) {
            memcpy(qr + sl * d, queries + (sl * m + r) * d, sizeof(double) * (size_t)d);
            memcpy(dor + (size_t)sl * per, d_o + ((size_t)sl * (size_t)m + (size_t)r) * per, sizeof(double) * per);
            memcpy(dlr + sl * T, d_lse + (sl * m + r) * T, sizeof(double) * (size_t)T);
        }
        rc = oracle_read_bwd_lse(ur, n_src, T, d, qr, S, gain, eps, dor, dlr, du, dqr, dgr);
        if (rc) break;
        for (int64_t sl = 0; sl < S; ++sl)
            memcpy(dqueries + (sl * m + r) * d, dqr + sl * d, sizeof(double) * (size_t)d);
        for (int64_t k = 0; k < d; ++k) dgain[k] += dgr[k];
        if (r == 0) {
            for (size_t k = 0; k < (size_t)n_src * per; ++k) dsrc[k] += du[k];
            continue;
        }
        const int64_t kr = ksizes[r - 1];
        for (int64_t i = 0; i < n_src; ++i)
            conv_transpose(src + (size_t)i * per, du + (size_t)i * per, T, d, kr, conv_w + off, dsrc + (size_t)i * per,
                           dconv_w + off);
        off += d * kr;
    }
    free(ue); free(ur); free(du); free(qr); free(dor); free(dlr); free(dqr); free(dgr);
    return rc;
}
