/*
 * spec_oracle.c -- CPU oracle for speculative-decoding verify-and-accept.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, fp64 statement of
 * what the verification step computes.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may build or call it; the product path
 * (the CUDA library and its binding) never does.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * Sources (the speculative-decoding pages):
 *  - EAGLE-3 review, "Speculative Decoding" (draft / verification / accept or
 *    reject): target distributions at k+1 positions from one forward; check
 *    drafts front to back; stop at the first rejection; resample the rejected
 *    position; a bonus token when every draft is accepted.
 *  - EAGLE-3 review, "small model answers" section: greedy rule (accept iff
 *    the draft equals the target argmax, else emit the target argmax);
 *    A(x) = min(1, p(x)/q(x)); residual norm(max(0, p - q)); identity
 *    min(p,q) + max(0,p-q) = p.
 *  - EAGLE-3 review, "EAGLE-3 inference" steps 4-5: greedy trees keep the
 *    longest prefix that matches the target's choices; only the accepted
 *    path's KV is kept.
 *  - vLLM EAGLE walkthrough, "rejected tokens" / "slot mapping" sections:
 *    rejected positions' slot_mapping entries become PADDING_SLOT_ID.
 *  - serving-book chapter, "acceptance rule preserving the output
 *    distribution": temperature 0 means greedy.
 *  - vLLM EAGLE walkthrough, "slot mapping and KV-cache management" (the names
 *    of the next-step preparation helpers) and the EAGLE-3 review, "EAGLE-3
 *    inference" step 5 (keep only the accepted path's KV, then draft again
 *    from the confirmed prefix): next-step inputs and tree KV compaction.
 *  - serving-book chapter, table of draft sources, row "n-gram lookup": find,
 *    in the prompt or the text generated so far, a span equal to the current
 *    ending and propose what follows it (no model).
 *
 * Readings where the pages are silent (the same list is kept in the design
 * notes): ties in argmax go to the lowest vocabulary index; q is used as given
 * (no temperature applied to it); accept iff q(x) == 0 or u < p(x)/q(x); the
 * resample of a request rejected at position a consumes u_sample[b][a], the
 * bonus consumes u_sample[b][k]; the inverse CDF picks the smallest j whose
 * prefix sum exceeds t = u * (total mass); a residual of zero total mass falls
 * back to sampling from p; a draft token outside [0, V) is a rejection with
 * p(x) = 0; tree ties at equal depth go to the smallest node index.
 *
 * All arithmetic on probabilities is IEEE double, evaluated in index order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_BF16 0
#define OR_FP32 1

/* Flag windows for positions whose GPU result may legitimately differ. */
#define OR_ACCEPT_WINDOW 1e-6   /* |u - p/q| below this flags the accept test   */
#define OR_EDGE_WINDOW 1e-5     /* t within this fraction of a CDF edge flags it */

/* ---------------------------------------------------------------- values -- */

/* The real number a stored logit denotes.  bf16 is the upper half of an IEEE
 * binary32, so widening is a 16-bit shift of the bit pattern. */
static double logit_at(const void *z, int dtype, size_t idx)
{
    if (dtype == OR_BF16) {
        uint32_t w = (uint32_t)((const uint16_t *)z)[idx] << 16;
        float f;
        memcpy(&f, &w, sizeof f);
        return (double)f;
    }
    return (double)((const float *)z)[idx];
}

/* argmax over one row, first occurrence of the maximum wins. */
static int row_argmax(const void *z, int dtype, size_t off, int V)
{
    int best = 0;
    double bv = logit_at(z, dtype, off);
    for (int j = 1; j < V; ++j) {
        double v = logit_at(z, dtype, off + (size_t)j);
        if (v > bv) {
            bv = v;
            best = j;
        }
    }
    return best;
}

/* p_j = exp(s_j - max s) / sum_i exp(s_i - max s), s_j = z_j / T. */
static void row_softmax(const void *z, int dtype, size_t off, int V, double T, double *p)
{
    double m = -INFINITY;
    for (int j = 0; j < V; ++j) {
        p[j] = logit_at(z, dtype, off + (size_t)j) / T;
        if (p[j] > m)
            m = p[j];
    }
    double sum = 0.0;
    for (int j = 0; j < V; ++j) {
        p[j] = exp(p[j] - m);
        sum += p[j];
    }
    for (int j = 0; j < V; ++j)
        p[j] /= sum;
}

/* Inverse CDF over non-negative weights w: t = u * sum(w); the result is the
 * smallest j with C_j = w_0 + ... + w_j > t.  If rounding leaves t >= C_{V-1},
 * the last j with w_j > 0 is taken.  *near_edge reports whether t lies within
 * OR_EDGE_WINDOW (relative) of the bucket's lower or upper edge. */
static int inverse_cdf(const double *w, int V, double u, int *near_edge)
{
    double total = 0.0;
    for (int j = 0; j < V; ++j)
        total += w[j];
    double t = u * total;
    double c = 0.0;
    int last_pos = -1;
    for (int j = 0; j < V; ++j) {
        double lo = c;
        c += w[j];
        if (w[j] > 0.0)
            last_pos = j;
        if (c > t) {
            int flag = 0;
            if (lo > 0.0 && t - lo <= OR_EDGE_WINDOW * lo)
                flag = 1;
            if (c - t <= OR_EDGE_WINDOW * c)
                flag = 1;
            *near_edge = flag;
            return j;
        }
    }
    *near_edge = 1;
    return last_pos < 0 ? V - 1 : last_pos;
}

/* ------------------------------------------------------------- the chain -- */

typedef struct {
    const void *logits;
    int dtype;
    const float *q;
    const int32_t *tokens;
    const float *temperature;
    const float *u_accept;
    const float *u_sample;
    int B, k, V;
    int32_t *out_tokens;
    int32_t *out_num_accepted;
    int32_t *flag_accept; /* [B, k] or NULL: 1 where |u - p/q| < window */
    int32_t *flag_sample; /* [B] or NULL: 1 where the sampled token sits near an edge */
    double *b_alg;        /* [B] or NULL: bytes the method must read */
    double *accept_ratio; /* [B, k] or NULL: p(x)/q(x) per accept test (NaN if not run) */
    int nthreads;
    int next;             /* shared request counter */
    pthread_mutex_t lock;
} chain_job;

static void chain_one(chain_job *J, int b, double *p, double *r)
{
    const int k = J->k, V = J->V;
    const size_t zs = (J->dtype == OR_BF16) ? 2 : 4;
    const size_t row = (size_t)V;
    const size_t zbase = (size_t)b * (size_t)(k + 1) * row;
    const double T = (double)J->temperature[b];
    int32_t *out = J->out_tokens + (size_t)b * (size_t)(k + 1);
    for (int i = 0; i <= k; ++i)
        out[i] = -1;
    if (J->flag_accept)
        for (int i = 0; i < k; ++i)
            J->flag_accept[(size_t)b * k + i] = 0;
    if (J->accept_ratio)
        for (int i = 0; i < k; ++i)
            J->accept_ratio[(size_t)b * k + i] = NAN;
    if (J->flag_sample)
        J->flag_sample[b] = 0;

    int a = k;
    double bytes = 0.0;
    if (T == 0.0) {
        /* greedy: accept while the draft equals the target argmax */
        for (int i = 0; i <= k; ++i) {
            int g = row_argmax(J->logits, J->dtype, zbase + (size_t)i * row, V);
            bytes += (double)row * (double)zs;
            if (i == k) {
                out[k] = g;
                a = k;
                break;
            }
            int x = J->tokens[(size_t)b * k + i];
            if (x != g) {
                out[i] = g;
                a = i;
                break;
            }
            out[i] = x;
        }
    } else {
        int sampled_row = -1; /* row whose distribution supplies the last token */
        int residual = 0;
        for (int i = 0; i < k; ++i) {
            row_softmax(J->logits, J->dtype, zbase + (size_t)i * row, V, T, p);
            bytes += (double)row * (double)zs;
            int x = J->tokens[(size_t)b * k + i];
            const float *qi = J->q + ((size_t)b * (size_t)k + (size_t)i) * row;
            int accept;
            if (x < 0 || x >= V) {
                accept = 0; /* out-of-range draft: p(x) = 0 */
            } else {
                double ph = p[x];
                double qh = (double)qi[x];
                bytes += 4.0;
                if (qh == 0.0) {
                    accept = 1;
                } else {
                    double ratio = ph / qh;
                    double u = (double)J->u_accept[(size_t)b * k + i];
                    accept = u < ratio;
                    if (J->accept_ratio)
                        J->accept_ratio[(size_t)b * k + i] = ratio;
                    if (J->flag_accept && fabs(u - ratio) < OR_ACCEPT_WINDOW)
                        J->flag_accept[(size_t)b * k + i] = 1;
                }
            }
            if (!accept) {
                a = i;
                sampled_row = i;
                residual = 1;
                /* residual r_j = max(0, p_j - q_j) */
                for (int j = 0; j < V; ++j) {
                    double d = p[j] - (double)qi[j];
                    r[j] = d > 0.0 ? d : 0.0;
                }
                bytes += (double)row * 4.0;
                break;
            }
            out[i] = x;
        }
        if (sampled_row < 0) {
            a = k;
            sampled_row = k;
            row_softmax(J->logits, J->dtype, zbase + (size_t)k * row, V, T, p);
            bytes += (double)row * (double)zs;
        }
        const double u = (double)J->u_sample[(size_t)b * (k + 1) + sampled_row];
        const double *w = p;
        if (residual) {
            double Z = 0.0;
            for (int j = 0; j < V; ++j)
                Z += r[j];
            if (Z > 0.0)
                w = r; /* zero residual mass: sample from p instead */
        }
        int edge = 0;
        out[sampled_row] = inverse_cdf(w, V, u, &edge);
        if (J->flag_sample)
            J->flag_sample[b] = edge;
    }
    J->out_num_accepted[b] = a;
    if (J->b_alg)
        J->b_alg[b] = bytes;
}

static void *chain_worker(void *arg)
{
    chain_job *J = (chain_job *)arg;
    double *p = (double *)malloc(sizeof(double) * (size_t)J->V);
    double *r = (double *)malloc(sizeof(double) * (size_t)J->V);
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int b = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (b >= J->B)
            break;
        chain_one(J, b, p, r);
    }
    free(p);
    free(r);
    return NULL;
}

/* Returns 0 on success, nonzero on bad arguments. */
int oracle_verify_chain(const void *logits, int dtype, const float *draft_probs,
                        const int32_t *draft_tokens, const float *temperature,
                        const float *u_accept, const float *u_sample, int B, int k, int V,
                        int32_t *out_tokens, int32_t *out_num_accepted, int32_t *flag_accept,
                        int32_t *flag_sample, double *b_alg, double *accept_ratio, int nthreads)
{
    /* k = 0 (a request with no drafts) emits the bonus token of row 0 */
    if (B < 0 || k < 0 || V < 1 || !logits || (k > 0 && !draft_tokens) || !temperature || !u_sample ||
        !out_tokens || !out_num_accepted)
        return 1;
    for (int b = 0; b < B; ++b)
        if (temperature[b] != 0.0f && (!draft_probs || !u_accept))
            return 1;
    chain_job J;
    memset(&J, 0, sizeof J);
    J.logits = logits;
    J.dtype = dtype;
    J.q = draft_probs;
    J.tokens = draft_tokens;
    J.temperature = temperature;
    J.u_accept = u_accept;
    J.u_sample = u_sample;
    J.B = B;
    J.k = k;
    J.V = V;
    J.out_tokens = out_tokens;
    J.out_num_accepted = out_num_accepted;
    J.flag_accept = flag_accept;
    J.flag_sample = flag_sample;
    J.b_alg = b_alg;
    J.accept_ratio = accept_ratio;
    J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > B)
        nthreads = B > 0 ? B : 1;
    if (nthreads == 1) {
        chain_worker(&J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int t = 0; t < nthreads; ++t)
            pthread_create(&th[t], NULL, chain_worker, &J);
        for (int t = 0; t < nthreads; ++t)
            pthread_join(th[t], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* -------------------------------------------------------------- the tree -- */

/* Greedy tree: g_n = argmax of row n; node n is accepted iff its parent is
 * accepted and token_n == g_{parent(n)}; the root (node 0) is accepted.  The
 * chosen node n* is the deepest accepted node (smallest index on ties); the
 * output is the path root..n*, the path's tokens, then g_{n*}. */
int oracle_verify_tree(const void *logits, int dtype, const int32_t *node_tokens,
                       const int32_t *parent, int B, int N, int V, int max_depth,
                       int32_t *out_path, int32_t *out_tokens, int32_t *out_len, double *b_alg)
{
    if (B < 0 || N < 0 || V < 1 || max_depth < 0 || !logits || !parent || !out_path ||
        !out_tokens || !out_len)
        return 1;
    if (N > 0 && !node_tokens)
        return 1;
    if (parent[0] != -1)
        return 1;
    int *depth = (int *)malloc(sizeof(int) * (size_t)(N + 1));
    int *g = (int *)malloc(sizeof(int) * (size_t)(N + 1));
    int *acc = (int *)malloc(sizeof(int) * (size_t)(N + 1));
    int *has_child = (int *)calloc((size_t)(N + 1), sizeof(int));
    depth[0] = 0;
    int bad = 0;
    for (int n = 1; n <= N; ++n) {
        if (parent[n] < 0 || parent[n] >= n) {
            bad = 1;
            break;
        }
        depth[n] = depth[parent[n]] + 1;
        if (depth[n] > max_depth)
            bad = 1;
        has_child[parent[n]] = 1;
    }
    if (!bad) {
        const size_t zs = (dtype == OR_BF16) ? 2 : 4;
        const size_t row = (size_t)V;
        for (int b = 0; b < B; ++b) {
            const size_t zbase = (size_t)b * (size_t)(N + 1) * row;
            for (int n = 0; n <= N; ++n)
                g[n] = row_argmax(logits, dtype, zbase + (size_t)n * row, V);
            acc[0] = 1;
            int best = 0;
            for (int n = 1; n <= N; ++n) {
                int x = node_tokens[(size_t)b * N + (n - 1)];
                acc[n] = acc[parent[n]] && x == g[parent[n]];
                if (acc[n] && depth[n] > depth[best])
                    best = n;
            }
            int d = depth[best];
            int32_t *path = out_path + (size_t)b * (size_t)(max_depth + 1);
            int32_t *tok = out_tokens + (size_t)b * (size_t)(max_depth + 1);
            for (int i = 0; i <= max_depth; ++i) {
                path[i] = -1;
                tok[i] = -1;
            }
            for (int n = best, i = d; i >= 0; n = parent[n], --i)
                path[i] = n;
            for (int i = 1; i <= d; ++i)
                tok[i - 1] = node_tokens[(size_t)b * N + (path[i] - 1)];
            tok[d] = g[best];
            out_len[b] = d + 1;
            if (b_alg) {
                double rows = 0.0;
                for (int n = 0; n <= N; ++n)
                    if (n == 0 || n == best || (acc[n] && has_child[n]))
                        rows += 1.0;
                b_alg[b] = rows * (double)row * (double)zs;
            }
        }
    }
    free(depth);
    free(g);
    free(acc);
    free(has_child);
    return bad ? 1 : 0;
}

/* ------------------------------------------------------ the sampled tree -- */

/* Sampled token tree (EAGLE-3 review, "EAGLE-3 inference" step 4: sampling
 * keeps min(1, p/q) acceptance with residual correction; the pages give no
 * rule for siblings).  Reading taken: walk from the root; at node c the target
 * distribution is p' = softmax(z_c / T); the children of c are tested in index
 * order, child n with token x accepted iff q_c(x) == 0 or u_accept[n] <
 * p'(x) / q_c(x), where q_c (row c of draft_probs) is the distribution the
 * children of c were drawn from.  An accepted child becomes the next node; a
 * rejected one replaces p' by norm(max(0, p' - q_c)) (unchanged if that has
 * zero mass) before the next sibling.  When no child is accepted, or c is a
 * leaf, one token is drawn from p' by inverse CDF with u_sample[c].  A child
 * token outside [0, V) is rejected (p'(x) = 0).  With children drawn i.i.d.
 * from q_c this emits each token with law p (the chain's identity applied once
 * per sibling).
 *
 * Flag windows: the accept test's ratio and the inverse CDF's edges carry the
 * rounding of every term that went into them before the clip, so the windows
 * scale with g, the running "gross" value that starts at p and becomes
 * (g + q_c) / Z wherever a residual step keeps a positive entry (Z the
 * residual's mass): |u - ratio| < 1e-6 * max(1, g(x) / q_c(x)) flags a test,
 * and t within 1e-5 of the gross prefix sum of a bucket edge flags a draw.
 * With no residual step (g = p) these are the chain's windows. */
int oracle_verify_tree_sampled(const void *logits, int dtype, const float *draft_probs,
                               const int32_t *node_tokens, const int32_t *parent, const float *temperature,
                               const float *u_accept, const float *u_sample, int B, int N, int V,
                               int max_depth, int32_t *out_path, int32_t *out_tokens, int32_t *out_len,
                               int32_t *flag_accept, int32_t *flag_sample, double *b_alg)
{
    if (B < 0 || N < 0 || V < 1 || max_depth < 0 || !logits || !parent || !temperature || !u_sample ||
        !out_path || !out_tokens || !out_len)
        return 1;
    if (N > 0 && (!node_tokens || !draft_probs || !u_accept))
        return 1;
    if (parent[0] != -1)
        return 1;
    for (int b = 0; b < B; ++b)
        if (!(temperature[b] > 0.0f))
            return 1;
    int *depth = (int *)malloc(sizeof(int) * (size_t)(N + 1));
    int bad = 0;
    depth[0] = 0;
    for (int n = 1; n <= N; ++n) {
        if (parent[n] < 0 || parent[n] >= n) {
            bad = 1;
            break;
        }
        depth[n] = depth[parent[n]] + 1;
        if (depth[n] > max_depth)
            bad = 1;
    }
    if (bad) {
        free(depth);
        return 1;
    }
    const size_t zs = (dtype == OR_BF16) ? 2 : 4;
    const size_t row = (size_t)V;
    double *w = (double *)malloc(sizeof(double) * row);
    double *g = (double *)malloc(sizeof(double) * row);
    for (int b = 0; b < B; ++b) {
        const size_t zbase = (size_t)b * (size_t)(N + 1) * row;
        const double T = (double)temperature[b];
        int32_t *path = out_path + (size_t)b * (size_t)(max_depth + 1);
        int32_t *tok = out_tokens + (size_t)b * (size_t)(max_depth + 1);
        for (int i = 0; i <= max_depth; ++i) {
            path[i] = -1;
            tok[i] = -1;
        }
        if (flag_accept)
            for (int n = 0; n < N; ++n)
                flag_accept[(size_t)b * N + n] = 0;
        double bytes = 0.0;
        int c = 0, d = 0;
        path[0] = 0;
        for (;;) {
            row_softmax(logits, dtype, zbase + (size_t)c * row, V, T, w);
            bytes += (double)row * (double)zs;
            for (size_t j = 0; j < row; ++j)
                g[j] = w[j];
            const float *qc = draft_probs ? draft_probs + ((size_t)b * (size_t)(N + 1) + (size_t)c) * row : NULL;
            int next = -1, q_read = 0;
            for (int n = c + 1; n <= N && next < 0; ++n) {
                if (parent[n] != c)
                    continue;
                const int x = node_tokens[(size_t)b * N + (n - 1)];
                int accept = 0;
                if (x >= 0 && x < V) {
                    const double qh = (double)qc[x];
                    bytes += 4.0;
                    if (qh == 0.0) {
                        accept = 1;
                    } else {
                        const double ratio = w[x] / qh;
                        const double u = (double)u_accept[(size_t)b * N + (n - 1)];
                        accept = ratio > u;
                        double scale = g[x] / qh;
                        if (scale < 1.0)
                            scale = 1.0;
                        if (flag_accept && fabs(u - ratio) < OR_ACCEPT_WINDOW * scale)
                            flag_accept[(size_t)b * N + (n - 1)] = 1;
                    }
                }
                if (accept) {
                    next = n;
                    break;
                }
                /* p' <- norm(max(0, p' - q_c)); kept as it is if the residual has no mass */
                if (!q_read) {
                    bytes += (double)row * 4.0;
                    q_read = 1;
                }
                double Z = 0.0;
                for (size_t j = 0; j < row; ++j) {
                    const double r = w[j] - (double)qc[j];
                    Z += r > 0.0 ? r : 0.0;
                }
                if (Z > 0.0)
                    for (size_t j = 0; j < row; ++j) {
                        const double r = w[j] - (double)qc[j];
                        if (r > 0.0) {
                            w[j] = r / Z;
                            g[j] = (g[j] + (double)qc[j]) / Z;
                        } else {
                            w[j] = 0.0;
                            g[j] = 0.0;
                        }
                    }
            }
            if (next < 0)
                break;
            tok[d] = node_tokens[(size_t)b * N + (next - 1)];
            ++d;
            path[d] = next;
            c = next;
        }
        /* one draw from p' of the last node: smallest j with prefix above t */
        const double u = (double)u_sample[(size_t)b * (size_t)(N + 1) + (size_t)c];
        double total = 0.0;
        for (size_t j = 0; j < row; ++j)
            total += w[j];
        const double t = u * total;
        double cw = 0.0, cg = 0.0;
        int pick = -1, last_pos = -1, edge = 1;
        for (int j = 0; j < V; ++j) {
            const double lo = cw, glo = cg;
            cw += w[j];
            cg += g[j];
            if (w[j] > 0.0)
                last_pos = j;
            if (cw > t) {
                edge = (lo > 0.0 && t - lo <= OR_EDGE_WINDOW * glo) || (cw - t <= OR_EDGE_WINDOW * cg);
                pick = j;
                break;
            }
        }
        if (pick < 0)
            pick = last_pos < 0 ? V - 1 : last_pos;
        tok[d] = pick;
        out_len[b] = d + 1;
        if (flag_sample)
            flag_sample[b] = edge;
        if (b_alg)
            b_alg[b] = bytes;
    }
    free(w);
    free(g);
    free(depth);
    return 0;
}

/* ------------------------------------------------------------ slot fix-up -- */

/* Chain mode (path == NULL): entries j > num_accepted[b] become pad.
 * Tree mode: entry j survives iff j == 0 or j appears in path[b, :]. */
int oracle_fixup_slots(int64_t *slot_mapping, int B, int P, const int32_t *num_accepted,
                       const int32_t *path, int path_stride, int64_t pad)
{
    if (B < 0 || P < 0 || !slot_mapping)
        return 1;
    if (!num_accepted && !path)
        return 1;
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < P; ++j) {
            int keep;
            if (!path) {
                keep = j <= num_accepted[b];
            } else {
                keep = (j == 0);
                for (int i = 0; i < path_stride && !keep; ++i)
                    keep = path[(size_t)b * path_stride + i] == j;
            }
            if (!keep)
                slot_mapping[(size_t)b * P + j] = pad;
        }
    }
    return 0;
}

/* ---------------------------------------------------------- n-gram lookup -- */

/* For each sequence s[0..L-1] (row b of tokens, L = lengths[b]): the longest
 * n in [n_min, n_max] for which the ending s[L-n..L-1] also occurs ending at
 * an earlier position e < L-1 (s[e-n+1..e] == s[L-n..L-1]); among the
 * occurrences of that length the latest (largest e).  The draft is the tokens
 * after it, s[e+1..], at most k of them (fewer if the text ends first).
 * No such n: no draft (count 0, match_len 0, match_end -1).  Readings (the
 * page is silent): longest n first, then the most recent occurrence. */
int oracle_ngram_propose(const int32_t *tokens, const int32_t *lengths, int B, int Lmax, int n_min, int n_max,
                         int k, int32_t *out_draft, int32_t *out_count, int32_t *out_match_len,
                         int32_t *out_match_end)
{
    if (B < 0 || Lmax < 0 || n_min < 1 || n_max < n_min || k < 0 || !out_draft || !out_count)
        return 1;
    for (int b = 0; b < B; ++b) {
        const int32_t *s = tokens + (size_t)b * Lmax;
        int L = lengths[b];
        if (L < 0 || L > Lmax)
            return 1;
        int best_n = 0, best_e = -1;
        for (int n = n_max; n >= n_min && best_e < 0; --n) {
            if (n > L - 1)
                continue;  /* the ending and an earlier copy need n + 1 tokens at least */
            for (int e = L - 2; e >= n - 1; --e) {
                int same = 1;
                for (int t = 0; t < n && same; ++t)
                    same = s[e - t] == s[L - 1 - t];
                if (same) {
                    best_n = n;
                    best_e = e;
                    break;
                }
            }
        }
        int count = 0;
        for (int j = 0; j < k; ++j) {
            int32_t v = -1;
            if (best_e >= 0 && best_e + 1 + j < L) {
                v = s[best_e + 1 + j];
                ++count;
            }
            out_draft[(size_t)b * k + j] = v;
        }
        out_count[b] = count;
        if (out_match_len)
            out_match_len[b] = best_n;
        if (out_match_end)
            out_match_end[b] = best_e;
    }
    return 0;
}

/* -------------------------------------------------- next-step preparation -- */

/* After verification of request b (row 0 at sequence position positions[b],
 * rows 0..k at positions[b]..positions[b]+k, a = num_accepted[b] drafts
 * accepted), the token emitted last, out_tokens[b][a], is the next step's
 * first input, at position positions[b] + a + 1.  Readings (the pages give
 * only the helpers' names): the next step writes P_next rows at positions
 * next_position .. next_position + P_next - 1, whose KV slots come from the
 * block table, slot = block_table[b][pos / block_size] * block_size +
 * pos % block_size, or pad when pos / block_size is past the table or the
 * entry is negative (status bit 1); the drafter's hidden-state input is the
 * target's row of the last accepted position, flat row index
 * row0(b) + a, row0(b) = b * rows_per_req (padded) or cu[b] + b (ragged);
 * that row of hidden_in (row_bytes bytes) is copied to hidden_out[b]. */
int oracle_prepare_next_step(const int32_t *out_tokens, int out_stride, const int32_t *num_accepted,
                             const int32_t *positions, const int32_t *block_table, int max_blocks,
                             int block_size, int B, int P_next, int rows_per_req, const int32_t *cu,
                             const uint8_t *hidden_in, int64_t row_bytes, int64_t pad, int32_t *next_token,
                             int32_t *next_position, int64_t *next_slots, int32_t *last_row,
                             uint8_t *hidden_out, int32_t *status)
{
    if (B < 0 || out_stride < 1 || max_blocks < 0 || block_size < 1 || P_next < 0 || !out_tokens ||
        !num_accepted || !positions || !next_token || !next_position)
        return 1;
    if (P_next > 0 && (!block_table || !next_slots))
        return 1;
    if (!cu && rows_per_req < 1)
        return 1;
    if (hidden_in && (!hidden_out || row_bytes < 1))
        return 1;
    int st = 0;
    for (int b = 0; b < B; ++b) {
        const int a = num_accepted[b];
        if (a < 0 || a >= out_stride)
            return 1;
        next_token[b] = out_tokens[(size_t)b * out_stride + a];
        const int64_t np = (int64_t)positions[b] + a + 1;
        next_position[b] = (int32_t)np;
        for (int j = 0; j < P_next; ++j) {
            const int64_t pos = np + j;
            const int64_t blk = pos / block_size;
            int64_t slot = pad;
            if (blk < max_blocks) {
                const int32_t e = block_table[(size_t)b * max_blocks + blk];
                if (e >= 0)
                    slot = (int64_t)e * block_size + pos % block_size;
                else
                    st |= 1;
            } else {
                st |= 1;
            }
            next_slots[(size_t)b * P_next + j] = slot;
        }
        const int64_t r0 = cu ? (int64_t)cu[b] + b : (int64_t)b * rows_per_req;
        const int64_t r = r0 + a;
        if (last_row)
            last_row[b] = (int32_t)r;
        if (hidden_in)
            memcpy(hidden_out + (size_t)b * (size_t)row_bytes, hidden_in + (size_t)r * (size_t)row_bytes,
                   (size_t)row_bytes);
    }
    if (status)
        *status |= st;
    return 0;
}

/* Tree KV compaction: the accepted path root = n_0, n_1, ..., n_d
 * (d = out_len[b] - 1) was verified with node n's KV in slot
 * slot_mapping[b][n]; afterwards depth i of the path must sit where the chain
 * keeps position i, slot_mapping[b][i].  Every destination slot receives the
 * row its source slot held before the call (sources are read before any
 * destination is written).  A source or destination outside [0, num_slots)
 * is skipped with status bit 1. */
int oracle_compact_tree_kv(uint8_t *kv, int64_t num_slots, int64_t row_bytes, const int64_t *slot_mapping,
                           int slot_stride, const int32_t *path, int path_stride, const int32_t *out_len, int B,
                           int32_t *status)
{
    if (B < 0 || num_slots < 0 || row_bytes < 1 || slot_stride < 1 || path_stride < 1 || !kv || !slot_mapping ||
        !path || !out_len)
        return 1;
    int st = 0;
    uint8_t *tmp = (uint8_t *)malloc((size_t)row_bytes * (size_t)path_stride);
    int64_t *dst = (int64_t *)malloc(sizeof(int64_t) * (size_t)path_stride);
    for (int b = 0; b < B; ++b) {
        const int L = out_len[b];
        if (L < 1 || L > path_stride || L > slot_stride) {
            free(tmp);
            free(dst);
            return 1;
        }
        int nmove = 0;
        for (int i = 1; i < L; ++i) {
            const int node = path[(size_t)b * path_stride + i];
            if (node < 0 || node >= slot_stride) {
                st |= 1;
                continue;
            }
            if (node == i)
                continue;
            const int64_t s_src = slot_mapping[(size_t)b * slot_stride + node];
            const int64_t s_dst = slot_mapping[(size_t)b * slot_stride + i];
            if (s_src < 0 || s_src >= num_slots || s_dst < 0 || s_dst >= num_slots) {
                st |= 1;
                continue;
            }
            memcpy(tmp + (size_t)nmove * (size_t)row_bytes, kv + (size_t)s_src * (size_t)row_bytes, (size_t)row_bytes);
            dst[nmove++] = s_dst;
        }
        for (int i = 0; i < nmove; ++i)
            memcpy(kv + (size_t)dst[i] * (size_t)row_bytes, tmp + (size_t)i * (size_t)row_bytes, (size_t)row_bytes);
    }
    free(tmp);
    free(dst);
    if (status)
        *status |= st;
    return 0;
}
