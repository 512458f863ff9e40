/*
 * specv_oracle.c -- plain, slow, fp64 CPU oracle for the speculative-decoding
 * verify/accept step with RAPID's inference-time knowledge transfer.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the CPU-baseline
 * leg of the benchmark call this file; the CUDA library never includes, links
 * or calls it, and it includes nothing of the CUDA library.
 *
 * Sources (page title, then section):
 *   [RAPID]  "RAPID：基于检索增强的推测解码长上下文推理"
 *            (papers.ananclaw.com explainer of arXiv 2502.20330)
 *            - "核心方法 / 2) 推理时知识迁移": the displayed mixture equation
 *              p~ = (1-lambda) p_t + lambda p_q;
 *            - "核心方法 / 3) 候选验证机制（伪代码）": the per-step loop:
 *              softmax of the enhanced target row and of the draft row,
 *              r ~ U(0,1), accept iff r < min(1, p~(x)/p_q(x)), otherwise
 *              resample and stop.
 *   [SD]     "大模型推理的Speculative Decoding原理详解"
 *            - "数学原理 / 修改的拒绝采样": accept with probability
 *              min(1, p/q), otherwise resample from the (p - q) distribution
 *              and discard the rest of the draft.
 *   [EAGLE]  "投机解码（EAGLE）：让小模型猜、大模型验，无损加速 LLM 生成"
 *            - "关键技术点 / 1. 为什么无损": the resample distribution is
 *              max(0, p - q) (normalised), which makes the output exact;
 *            - "核心思路", step 3 (accept/reject): a draft token that is the
 *              target model's most likely token is accepted outright (the
 *              greedy clause).
 *
 * Readings taken where the pages are silent or ambiguous (each one is also
 * listed in the design notes):
 *   - The RAPID pseudocode prints the resample as sample(p_t - p_q); the
 *     distribution used is normalize(max(0, p~ - q)) as in [EAGLE] and [SD].
 *   - The comparison is strict (r < accept_prob): an exact tie rejects.
 *   - When all K drafts are accepted one bonus token is drawn from p~ at
 *     position K+1, and p~ there equals the target softmax (no draft row
 *     exists at K+1, so lambda has nothing to mix).
 *   - One uniform u_resample per sequence serves the resample or the bonus
 *     (only one of them happens per sequence).
 *   - Inverse CDF: the smallest v whose inclusive prefix sum, summed
 *     sequentially in index order, is strictly greater than u * W.  If none
 *     is (round-off), the largest v with positive weight.
 *   - If the residual has zero mass (possible only through round-off) the
 *     token is drawn from p~ of the same row instead.
 *   - q(x) = 0: the ratio is +infinity (accept) unless p~(x) = 0 too, which
 *     rejects.
 *   - Invalid input (a draft token outside [0, V), or lambda outside [0, 1]
 *     or NaN) gives n_accepted = -1 and all output tokens -1.
 *
 *   - Masked logits (-inf: a padded vocabulary, a grammar or top-k mask) in
 *     the logit mixture (1 - lambda) z_t + lambda z_q: a masked entry of a
 *     row whose weight is positive masks the mixed entry, and a term of
 *     weight zero drops out (so lambda = 0 gives z_t and lambda = 1 gives
 *     z_q whatever the other row holds).
 *   - Greedy verification (the greedy clause of [EAGLE] "核心思路") is read as:
 *     accept x_i iff x_i is the argmax of the mixed logits
 *     w = (1 - lambda) z_t + lambda z_q of row i (the logit-space enhanced
 *     target, whose softmax is p~ in logit mode; lambda = 0 gives the
 *     target's own argmax, the clause as printed), emit that argmax at the
 *     first mismatch, and the argmax of target row K when every draft
 *     matches.  Equal maxima go to the smallest index.  w is formed in
 *     double precision like everything else; for each decided mixed row the
 *     oracle also reports the gap between the largest and the second largest
 *     w relative to the row's largest logit magnitude, so that a caller can
 *     tell which rows a lower-precision argmax may decide otherwise.
 *
 * Everything is computed in double precision.  fp32 inputs are promoted
 * exactly; bf16 inputs are widened to fp32 (exactly) by the caller first.
 * Build with -ffp-contract=off so no multiply-add is fused behind our back.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_PROB_MIX 0
#define ORACLE_LOGIT_MIX 1

/* bits of oracle_verify's per-sequence flags */
#define ORACLE_FLAG_INVALID 1          /* invalid input: outputs are -1 */
#define ORACLE_FLAG_RESIDUAL_ZERO 2    /* residual had zero mass: drew from p~ */
#define ORACLE_FLAG_CDF_FALLBACK 4     /* no prefix exceeded u*W: took the last positive */
#define ORACLE_FLAG_BONUS 8            /* every draft accepted: bonus token drawn */

/* ------------------------------------------------------------------------ */
/* softmax of one row: p_v = exp(z_v - max_u z_u) / sum_u exp(z_u - max_u z_u)
 * [RAPID] "3) 候选验证机制": softmax(enhanced_target[i]), softmax(draft_logits[i]). */
void oracle_softmax(const double *z, int64_t V, double *p)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
        if (z[v] > m) m = z[v];
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        p[v] = exp(z[v] - m);
        s += p[v];
    }
    for (int64_t v = 0; v < V; ++v) p[v] = p[v] / s;
}

/* probability-mode mixture p~ = (1 - lambda) * p_t + lambda * p_q
 * [RAPID] "2) 推理时知识迁移", displayed equation. */
void oracle_mix_prob(const double *pt, const double *pq, double lambda, int64_t V,
                     double *out)
{
    for (int64_t v = 0; v < V; ++v) out[v] = (1.0 - lambda) * pt[v] + lambda * pq[v];
}

/* One entry of the logit-space mixture (1 - lambda) * z_t + lambda * z_q
 * ([RAPID] "3) 候选验证机制": enhanced_target = (1-λ)*target_logits +
 * λ*draft_logits), with the masking reading of the header: a -inf logit whose
 * weight is positive gives -inf, a term of weight zero contributes nothing. */
double oracle_mix_logit_entry(double zt, double zq, double lambda)
{
    double a = 1.0 - lambda, b = lambda, w = 0.0;
    if (a > 0.0) {
        if (zt == -INFINITY) return -INFINITY;
        w += a * zt;
    }
    if (b > 0.0) {
        if (zq == -INFINITY) return -INFINITY;
        w += b * zq;
    }
    return w;
}

/* logit-mode mixture p~ = softmax((1 - lambda) * z_t + lambda * z_q)
 * [RAPID] "3) 候选验证机制": then p_t = softmax(enhanced_target[i]). */
void oracle_mix_logit(const double *zt, const double *zq, double lambda, int64_t V,
                      double *out)
{
    double *w = (double *)malloc((size_t)V * sizeof(double));
    for (int64_t v = 0; v < V; ++v) w[v] = oracle_mix_logit_entry(zt[v], zq[v], lambda);
    oracle_softmax(w, V, out);
    free(w);
}

/* Inverse-CDF draw from a nonnegative weight vector w over V entries with
 * the uniform u: the smallest v with (w_0 + ... + w_v) > u * W, where W is the
 * sum of all weights, both sums taken sequentially in index order.  If no
 * prefix exceeds u * W (round-off), the largest v with w_v > 0.  Returns -1
 * when W == 0.  *fallback is set to 1 when the round-off rule decided.
 * If margin is not NULL it receives min_k |u - C_k / W| over every boundary
 * C_k = w_0 + ... + w_k, the distance of u to the nearest CDF boundary. */
int64_t oracle_sample_inverse_cdf(const double *w, int64_t V, double u, int *fallback,
                                  double *margin)
{
    double W = 0.0;
    for (int64_t v = 0; v < V; ++v) W += w[v];
    if (fallback) *fallback = 0;
    if (margin) *margin = INFINITY;
    if (!(W > 0.0)) return -1;
    double t = u * W;
    double c = 0.0;
    int64_t chosen = -1;
    for (int64_t v = 0; v < V; ++v) {
        c += w[v];
        if (margin) {
            double d = fabs(u - c / W);
            if (d < *margin) *margin = d;
        }
        if (chosen < 0 && c > t) chosen = v;
    }
    if (chosen < 0) {
        for (int64_t v = V - 1; v >= 0; --v)
            if (w[v] > 0.0) { chosen = v; break; }
        if (fallback) *fallback = 1;
    }
    return chosen;
}

/* The enhanced target p~ and the draft distribution q of position i of one
 * sequence.  For i < K: q = softmax(z_q[i]) and p~ by the chosen mode.  For
 * i == K (the bonus position) there is no draft row: p~ = softmax(z_t[K]) and
 * q is left untouched. */
static void rows_at(const float *zt_seq, const float *zq_seq, int32_t K, int64_t V,
                    int32_t i, double lambda, int mode, double *zt, double *zq,
                    double *pt, double *pq, double *ptilde)
{
    for (int64_t v = 0; v < V; ++v) zt[v] = (double)zt_seq[(int64_t)i * V + v];
    if (i == K) {
        oracle_softmax(zt, V, ptilde);
        return;
    }
    for (int64_t v = 0; v < V; ++v) zq[v] = (double)zq_seq[(int64_t)i * V + v];
    oracle_softmax(zq, V, pq);
    if (mode == ORACLE_PROB_MIX) {
        oracle_softmax(zt, V, pt);
        oracle_mix_prob(pt, pq, lambda, V, ptilde);
    } else {
        oracle_mix_logit(zt, zq, lambda, V, ptilde);
    }
}

/* Exported: p~ rows [K+1][V] and q rows [K][V] of one sequence (test helper). */
void oracle_rows(const float *zt_seq, const float *zq_seq, int32_t K, int64_t V,
                 double lambda, int mode, double *ptilde_out, double *q_out)
{
    double *zt = (double *)malloc((size_t)V * sizeof(double));
    double *zq = (double *)malloc((size_t)V * sizeof(double));
    double *pt = (double *)malloc((size_t)V * sizeof(double));
    for (int32_t i = 0; i <= K; ++i)
        rows_at(zt_seq, zq_seq, K, V, i, lambda, mode, zt, zq, pt,
                i < K ? q_out + (int64_t)i * V : pt, ptilde_out + (int64_t)i * V);
    free(zt);
    free(zq);
    free(pt);
}

/* Diagnostics written per sequence when the pointers are not NULL:
 *   ratio[K]        p~(x_i) / q(x_i) for every position i < K (+inf if q = 0)
 *   ptilde_x[K]     p~(x_i);  q_x[K]: q(x_i)
 *   alpha[K]        sum_v min(p~_v, q_v), the exact acceptance probability
 *   accept_margin   min over decided positions of |u_i - min(1, ratio_i)|
 *   cdf_margin      distance of u_resample to the nearest boundary of the
 *                   CDF it was drawn from (+inf if no draw)
 *   flags           ORACLE_FLAG_* bits
 * All positions' ratios and alphas are computed (diagnostics), but the
 * decision itself follows the pages' loop and stops at the first reject. */
typedef struct {
    double *ratio;
    double *ptilde_x;
    double *q_x;
    double *alpha;
    double *accept_margin;
    double *cdf_margin;
    int32_t *flags;
} oracle_diag;

static void verify_one(const float *zt_seq, const float *zq_seq, const int32_t *tok,
                       const float *ua, float ur, float lam, int32_t K, int64_t V, int mode,
                       int32_t *out_tok, int32_t *out_n, oracle_diag *d, int64_t b,
                       double *zt, double *zq, double *pt, double *pq, double *ptilde,
                       double *wbuf)
{
    int32_t flags = 0;
    double lambda = (double)lam;
    int invalid = !(lambda >= 0.0 && lambda <= 1.0);
    for (int32_t i = 0; i < K; ++i)
        if (tok[i] < 0 || (int64_t)tok[i] >= V) invalid = 1;
    if (d && d->accept_margin) d->accept_margin[b] = INFINITY;
    if (d && d->cdf_margin) d->cdf_margin[b] = INFINITY;
    if (invalid) {
        for (int32_t i = 0; i <= K; ++i) out_tok[i] = -1;
        *out_n = -1;
        if (d && d->flags) d->flags[b] = ORACLE_FLAG_INVALID;
        return;
    }

    /* Diagnostics over every position (not part of the decision). */
    if (d && (d->ratio || d->ptilde_x || d->q_x || d->alpha)) {
        for (int32_t i = 0; i < K; ++i) {
            rows_at(zt_seq, zq_seq, K, V, i, lambda, mode, zt, zq, pt, pq, ptilde);
            double px = ptilde[tok[i]], qx = pq[tok[i]];
            if (d->ptilde_x) d->ptilde_x[b * K + i] = px;
            if (d->q_x) d->q_x[b * K + i] = qx;
            if (d->ratio) d->ratio[b * K + i] = qx > 0.0 ? px / qx : (px > 0.0 ? INFINITY : 0.0);
            if (d->alpha) {
                double a = 0.0;
                for (int64_t v = 0; v < V; ++v) a += ptilde[v] < pq[v] ? ptilde[v] : pq[v];
                d->alpha[b * K + i] = a;
            }
        }
    }

    /* The pages' loop: for i in range(K): softmaxes, ratio, accept or
     * resample-and-break. */
    int32_t n = K;
    int64_t token = -1;
    double margin = INFINITY;
    for (int32_t i = 0; i < K; ++i) {
        rows_at(zt_seq, zq_seq, K, V, i, lambda, mode, zt, zq, pt, pq, ptilde);
        double px = ptilde[tok[i]], qx = pq[tok[i]];
        double accept_prob;
        if (qx > 0.0) {
            double ratio = px / qx;
            accept_prob = ratio < 1.0 ? ratio : 1.0;
        } else {
            accept_prob = px > 0.0 ? 1.0 : 0.0;
        }
        double u = (double)ua[i];
        double dm = fabs(u - accept_prob);
        if (dm < margin) margin = dm;
        if (u < accept_prob) {
            out_tok[i] = tok[i];
            continue;
        }
        /* Rejected at i: draw from normalize(max(0, p~ - q)). */
        n = i;
        for (int64_t v = 0; v < V; ++v) {
            double r = ptilde[v] - pq[v];
            wbuf[v] = r > 0.0 ? r : 0.0;
        }
        int fb = 0;
        double cm = INFINITY;
        token = oracle_sample_inverse_cdf(wbuf, V, (double)ur, &fb, &cm);
        if (token < 0) {
            /* zero residual mass (round-off only): draw from p~ instead */
            flags |= ORACLE_FLAG_RESIDUAL_ZERO;
            token = oracle_sample_inverse_cdf(ptilde, V, (double)ur, &fb, &cm);
        }
        if (fb) flags |= ORACLE_FLAG_CDF_FALLBACK;
        if (d && d->cdf_margin) d->cdf_margin[b] = cm;
        break;
    }
    if (n == K) {
        /* Every draft accepted: bonus token from p~ at position K+1, which is
         * the target softmax of row K. */
        rows_at(zt_seq, zq_seq, K, V, K, lambda, mode, zt, zq, pt, pq, ptilde);
        int fb = 0;
        double cm = INFINITY;
        token = oracle_sample_inverse_cdf(ptilde, V, (double)ur, &fb, &cm);
        if (fb) flags |= ORACLE_FLAG_CDF_FALLBACK;
        flags |= ORACLE_FLAG_BONUS;
        if (d && d->cdf_margin) d->cdf_margin[b] = cm;
    }
    out_tok[n] = (int32_t)token;
    for (int32_t i = n + 1; i <= K; ++i) out_tok[i] = -1;
    *out_n = n;
    if (d && d->accept_margin) d->accept_margin[b] = margin;
    if (d && d->flags) d->flags[b] = flags;
}

/* Verify sequences [b0, b1) of a batch.
 *   zt  [B][K+1][V] fp32 target logits      zq [B][K][V] fp32 draft logits
 *   tok [B][K] draft tokens                 ua [B][K] acceptance uniforms
 *   ur  [B] resample/bonus uniforms         lam [B] mixing coefficients
 *   out_tok [B][K+1], out_n [B]
 * Diagnostic arrays are indexed by the global sequence index b.
 * Returns 0, or -1 on allocation failure. */
int oracle_verify(const float *zt, const float *zq, const int32_t *tok, const float *ua,
                  const float *ur, const float *lam, int64_t b0, int64_t b1, int32_t K,
                  int64_t V, int mode, int32_t *out_tok, int32_t *out_n, double *ratio,
                  double *ptilde_x, double *q_x, double *alpha, double *accept_margin,
                  double *cdf_margin, int32_t *flags)
{
    oracle_diag d = {ratio, ptilde_x, q_x, alpha, accept_margin, cdf_margin, flags};
    double *buf = (double *)malloc((size_t)6 * (size_t)V * sizeof(double));
    if (!buf) return -1;
    double *zt_d = buf, *zq_d = buf + V, *pt = buf + 2 * V, *pq = buf + 3 * V;
    double *ptilde = buf + 4 * V, *wbuf = buf + 5 * V;
    for (int64_t b = b0; b < b1; ++b) {
        verify_one(zt + b * (int64_t)(K + 1) * V, zq + b * (int64_t)K * V, tok + b * K,
                   ua + b * K, ur[b], lam[b], K, V, mode, out_tok + b * (K + 1), out_n + b,
                   &d, b, zt_d, zq_d, pt, pq, ptilde, wbuf);
    }
    free(buf);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Greedy verification (reading in the header).                              */

/* The greedy scores of one row: w_v = (1 - lambda) z_t + lambda z_q with
 * the masking rule (zq == NULL: w = z_t, the bonus position). */
void oracle_greedy_scores(const float *zt, const float *zq, float lam, int64_t V, double *w)
{
    for (int64_t v = 0; v < V; ++v)
        w[v] = zq ? oracle_mix_logit_entry((double)zt[v], (double)zq[v], (double)lam)
                  : (double)zt[v];
}

/* Argmax over v of w_v, the first index among equal maxima.  If rel_gap is
 * not NULL it receives (w_best - w_second) / A, where w_second is the largest
 * w at any other index and A the largest finite |z_t|, |z_q| of the row: how
 * far the decision is from a tie, on the scale of the rounding error of a
 * lower-precision w (0 for an exact tie or an all-zero row, +inf when every
 * other entry is masked). */
int64_t oracle_greedy_argmax(const float *zt, const float *zq, float lam, int64_t V,
                             double *rel_gap)
{
    int64_t best = 0;
    double bw = -INFINITY, second = -INFINITY, A = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double w = zq ? oracle_mix_logit_entry((double)zt[v], (double)zq[v], (double)lam)
                      : (double)zt[v];
        if (v == 0 || w > bw) {
            if (v > 0) second = bw;
            bw = w;
            best = v;
        } else if (w > second) {
            second = w;
        }
        double at = fabs((double)zt[v]);
        if (at != INFINITY && at > A) A = at;
        if (zq) {
            double aq = fabs((double)zq[v]);
            if (aq != INFINITY && aq > A) A = aq;
        }
    }
    if (rel_gap) {
        if (V < 2 || second == -INFINITY)
            *rel_gap = INFINITY;
        else if (bw == second || !(A > 0.0))
            *rel_gap = 0.0;
        else
            *rel_gap = (bw - second) / A;
    }
    return best;
}

/* Greedy verification of sequences [b0, b1); same layouts as oracle_verify.
 * Invalid input (token outside [0, V), lambda outside [0, 1] or NaN) gives
 * n_accepted = -1 and all tokens -1.  tie_margin [B] (or NULL) receives the
 * smallest rel_gap of oracle_greedy_argmax over the mixed rows the decision
 * read (rows 0 .. min(n, K-1)); the bonus row's w is z_t itself, exact in
 * any precision, and is left out (+inf when no row counts). */
void oracle_verify_greedy(const float *zt, const float *zq, const int32_t *tok, const float *lam,
                          int64_t b0, int64_t b1, int32_t K, int64_t V, int32_t *out_tok,
                          int32_t *out_n, double *tie_margin)
{
    for (int64_t b = b0; b < b1; ++b) {
        const float *zt_b = zt + b * (int64_t)(K + 1) * V;
        const float *zq_b = zq + b * (int64_t)K * V;
        const int32_t *tk = tok + b * K;
        int32_t *ot = out_tok + b * (K + 1);
        double lambda = (double)lam[b];
        double margin = INFINITY;
        int invalid = !(lambda >= 0.0 && lambda <= 1.0);
        for (int32_t i = 0; i < K; ++i)
            if (tk[i] < 0 || (int64_t)tk[i] >= V) invalid = 1;
        if (invalid) {
            for (int32_t i = 0; i <= K; ++i) ot[i] = -1;
            out_n[b] = -1;
            if (tie_margin) tie_margin[b] = margin;
            continue;
        }
        int32_t n = K;
        int64_t token = -1;
        for (int32_t i = 0; i < K; ++i) {
            double g = INFINITY;
            int64_t a = oracle_greedy_argmax(zt_b + (int64_t)i * V, zq_b + (int64_t)i * V, lam[b],
                                             V, &g);
            if (g < margin) margin = g;
            if (a != (int64_t)tk[i]) {
                n = i;
                token = a;
                break;
            }
            ot[i] = tk[i];
        }
        if (n == K) token = oracle_greedy_argmax(zt_b + (int64_t)K * V, NULL, lam[b], V, NULL);
        ot[n] = (int32_t)token;
        for (int32_t i = n + 1; i <= K; ++i) ot[i] = -1;
        out_n[b] = n;
        if (tie_margin) tie_margin[b] = margin;
    }
}

/* ------------------------------------------------------------------------ */
/* Tree verification.
 *
 * Reading (the pages describe draft trees -- the speculative-decoding
 * explainer's "Tree Speculation" section: several candidate branches per
 * position, verified at once, so that another branch can be accepted when one
 * is rejected; the EAGLE explainer's "3. 验证阶段树形attention" and EAGLE-2's
 * dynamic draft tree -- but give no multi-branch acceptance rule).  A sequence's tree has nodes 0..N; node 0 is the root (the
 * last accepted position), node j >= 1 has parent[j] in [0, j) and token x_j.
 * Every node u has a target row z_t[u] (the target's next-token logits after
 * the path root..u) and, when draft_row[u] >= 0, the draft row
 * z_q[draft_row[u]] from which u's children were drawn, independently.  The
 * enhanced target at u is p~_u = mix(p_t[u], q_u) (the chosen mixture mode),
 * or p_t[u] when u has no draft row.  The walk, from u = 0:
 *   - p = p~_u; for each child c of u in index order: accept x_c iff
 *     u_accept[c] < min(1, p(x_c) / q_u(x_c)); on acceptance emit x_c and
 *     continue the walk at c; on rejection p = normalize(max(0, p - q_u));
 *   - if every child is rejected, draw the token from p (inverse CDF with
 *     u_resample); if u has no children, draw the bonus token from p~_u;
 *   - if a residual has zero mass (round-off only), draw from p~_u instead.
 * With one child per node (parent[j] = j - 1) this is the chain loop of
 * oracle_verify.  Invalid input: parent[0] != -1, parent[j] outside [0, j),
 * draft_row outside [-1, M), a node with children but no draft row, a token
 * outside [0, V), lambda outside [0, 1] -> n = -1, all outputs -1.
 */
static int tree_valid(const int32_t *par, const int32_t *drow, const int32_t *tok, int32_t N,
                      int32_t M, int64_t V, double lambda)
{
    if (!(lambda >= 0.0 && lambda <= 1.0)) return 0;
    if (par[0] != -1) return 0;
    for (int32_t j = 0; j <= N; ++j) {
        if (drow[j] < -1 || drow[j] >= M) return 0;
        if (j == 0) continue;
        if (par[j] < 0 || par[j] >= j) return 0;
        if (tok[j] < 0 || (int64_t)tok[j] >= V) return 0;
        if (drow[par[j]] < 0) return 0;
    }
    return 1;
}

/* p~ and q of node u (q left untouched when u has no draft row). */
static void tree_rows(const float *zt_seq, const float *zq_seq, const int32_t *drow, int64_t V,
                      int32_t u, double lambda, int mode, double *zt, double *zq, double *pt,
                      double *pq, double *ptilde)
{
    const float *rt = zt_seq + (int64_t)u * V;
    for (int64_t v = 0; v < V; ++v) zt[v] = (double)rt[v];
    if (drow[u] < 0) {
        oracle_softmax(zt, V, ptilde);
        return;
    }
    const float *rq = zq_seq + (int64_t)drow[u] * V;
    for (int64_t v = 0; v < V; ++v) zq[v] = (double)rq[v];
    oracle_softmax(zq, V, pq);
    if (mode == 0) {
        oracle_softmax(zt, V, pt);
        oracle_mix_prob(pt, pq, lambda, V, ptilde);
    } else {
        oracle_mix_logit(zt, zq, lambda, V, ptilde);
    }
}

/* Tree verification of sequences [b0, b1).
 *   zt  [B][N+1][V]   zq [B][M][V]   parent, draft_row, tok, ua: [B][N+1]
 *   ur, lam: [B]; out_tok, out_path: [B][N+1]; out_n: [B]
 *   accept_margin, cdf_margin: [B] or NULL (as for oracle_verify).
 * Returns 0, or -1 on allocation failure. */
int oracle_verify_tree(const float *zt, const float *zq, const int32_t *parent,
                       const int32_t *draft_row, const int32_t *tok, const float *ua,
                       const float *ur, const float *lam, int64_t b0, int64_t b1, int32_t N,
                       int32_t M, int64_t V, int mode, int32_t *out_tok, int32_t *out_path,
                       int32_t *out_n, double *accept_margin, double *cdf_margin)
{
    double *buf = (double *)malloc((size_t)6 * (size_t)V * sizeof(double));
    if (!buf) return -1;
    double *zt_d = buf, *zq_d = buf + V, *pt = buf + 2 * V, *pq = buf + 3 * V;
    double *ptilde = buf + 4 * V, *p = buf + 5 * V;
    for (int64_t b = b0; b < b1; ++b) {
        const float *zt_b = zt + b * (int64_t)(N + 1) * V;
        const float *zq_b = zq + b * (int64_t)M * V;
        const int32_t *par = parent + b * (N + 1), *drow = draft_row + b * (N + 1);
        const int32_t *tk = tok + b * (N + 1);
        const float *u_b = ua + b * (N + 1);
        int32_t *ot = out_tok + b * (N + 1), *op = out_path + b * (N + 1);
        for (int32_t j = 0; j <= N; ++j) ot[j] = op[j] = -1;
        double am = INFINITY, cm = INFINITY;
        double lambda = (double)lam[b];
        if (!tree_valid(par, drow, tk, N, M, V, lambda)) {
            out_n[b] = -1;
            if (accept_margin) accept_margin[b] = am;
            if (cdf_margin) cdf_margin[b] = cm;
            continue;
        }
        int32_t u = 0, n = 0;
        int64_t token = -1;
        for (;;) {
            tree_rows(zt_b, zq_b, drow, V, u, lambda, mode, zt_d, zq_d, pt, pq, ptilde);
            for (int64_t v = 0; v < V; ++v) p[v] = ptilde[v];
            int32_t next = -1, any_child = 0, exhausted = 0;
            for (int32_t c = u + 1; c <= N; ++c) {
                if (par[c] != u) continue;
                any_child = 1;
                double px = p[tk[c]], qx = pq[tk[c]];
                double accept_prob = qx > 0.0 ? (px / qx < 1.0 ? px / qx : 1.0)
                                              : (px > 0.0 ? 1.0 : 0.0);
                double dm = fabs((double)u_b[c] - accept_prob);
                if (dm < am) am = dm;
                if ((double)u_b[c] < accept_prob) {
                    next = c;
                    break;
                }
                /* rejected: p = normalize(max(0, p - q_u)) */
                double z = 0.0;
                for (int64_t v = 0; v < V; ++v) {
                    double r = p[v] - pq[v];
                    p[v] = r > 0.0 ? r : 0.0;
                    z += p[v];
                }
                if (!(z > 0.0)) {
                    exhausted = 1;
                    break;
                }
                for (int64_t v = 0; v < V; ++v) p[v] /= z;
            }
            if (next >= 0) {
                ot[n] = tk[next];
                op[n] = next;
                ++n;
                u = next;
                continue;
            }
            int fb = 0;
            /* no child: bonus from p~_u; every child rejected: the residual p;
             * a residual of zero mass: p~_u */
            const double *w = (!any_child || exhausted) ? ptilde : p;
            token = oracle_sample_inverse_cdf(w, V, (double)ur[b], &fb, &cm);
            break;
        }
        ot[n] = (int32_t)token;
        out_n[b] = n;
        if (accept_margin) accept_margin[b] = am;
        if (cdf_margin) cdf_margin[b] = cm;
    }
    free(buf);
    return 0;
}
