/*
 * oracle.c -- plain, slow, obviously-correct fp64 CPU oracle for batched
 * speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * execute this file: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only through seeded synthetic inputs.
 *
 * What it computes (source: "Accelerating Sonar through speculation",
 * Perplexity blog, and the work it cites in its References,
 * "Fast Inference from Transformers via Speculative Decoding"):
 *
 *  - §"Speculative decoding": every prefix of the drafted candidates is
 *    scored and the longest accepted one is kept; n drafted tokens give at
 *    most n+1 emitted tokens.
 *  - §"Target-Draft": acceptance compares the full probability
 *    distributions of the draft and target models; the target logits after
 *    the accepted prefix are sampled for one more token.
 *  - The exact rule is the cited work's: accept draft token x with
 *    probability min(1, p(x)/q(x)); at the first rejection draw from
 *    norm(max(0, p - q)); after a full accept draw a bonus token from the
 *    target's last row.
 *  - §"EAGLE": Top-K candidates per node of a draft tree; the longest
 *    accepted root-to-leaf path plus one target token.  Children are tested
 *    one after another; after each rejection the target distribution becomes
 *    the normalised residual (recursive rejection sampling).
 *  - §"MTP" / §"MTP schedule for a single token": token t_{i+1} pairs with
 *    hidden state H_i; a kernel inserts the next tokens into their slots.
 *
 * Readings where the pages are silent (choices of this oracle, not statements
 * of the pages):
 *  - temperature T == 0 means greedy (argmax, ties to the lowest index);
 *  - top-p keeps, in (logit desc, index asc) order, each token whose
 *    preceding mass is < top_p; top_p >= 1 disables it;
 *  - accept iff u < p/q with u in [0,1); q(x) == 0 rejects;
 *  - inverse CDF: the smallest v with C(v) > u * C(V-1);
 *  - a zero residual falls back to p itself;
 *  - Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) with
 *    key = (seed lo, seed hi), counter = (request lo, position lo,
 *    purpose | round << 8, request hi), u = (word0 >> 8) * 2^-24.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_NONFINITE 2
#define ORC_ERR_TOKEN 4
#define ORC_ERR_PARENT 8
#define ORC_ERR_LENGTH 16

#define ORC_PURPOSE_ACCEPT 1
#define ORC_PURPOSE_RESIDUAL 2
#define ORC_PURPOSE_BONUS 3
#define ORC_PURPOSE_DRAFT 4

#define ORC_CHILD_WOR 0
#define ORC_CHILD_IID 1
#define ORC_CHILD_DET 2

/* ------------------------------------------------------------------ */
/* Philox4x32-10, written from the SC'11 paper's definition.          */
/* ------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

double orc_uniform(uint64_t seed, int64_t req, int64_t pos, int purpose, int round)
{
    uint32_t ctr[4], key[2], out[4];
    uint64_t r = (uint64_t)req;
    ctr[0] = (uint32_t)r;
    ctr[1] = (uint32_t)(uint64_t)pos;
    ctr[2] = (uint32_t)purpose | ((uint32_t)round << 8);
    ctr[3] = (uint32_t)(r >> 32);
    key[0] = (uint32_t)seed;
    key[1] = (uint32_t)(seed >> 32);
    orc_philox4x32_10(ctr, key, out);
    return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------ */
/* Row helpers                                                        */
/* ------------------------------------------------------------------ */

/* A row is valid when it has no NaN, no +inf and at least one finite entry. */
static int row_valid(const double* x, int V)
{
    int any_finite = 0;
    for (int v = 0; v < V; ++v) {
        if (isnan(x[v])) return 0;
        if (isinf(x[v]) && x[v] > 0) return 0;
        if (isfinite(x[v])) any_finite = 1;
    }
    return any_finite;
}

/* Argmax with ties to the lowest index, over entries that are neither NaN
 * nor +inf.  Returns 0 when no such entry exists. */
int orc_argmax(const double* x, int V)
{
    int best = -1;
    for (int v = 0; v < V; ++v) {
        if (isnan(x[v]) || (isinf(x[v]) && x[v] > 0)) continue;
        if (best < 0 || x[v] > x[best]) best = v;
    }
    return best < 0 ? 0 : best;
}

typedef struct { double x; int idx; } keyed;

static int keyed_cmp(const void* a, const void* b)
{
    const keyed* p = (const keyed*)a;
    const keyed* q = (const keyed*)b;
    if (p->x > q->x) return -1;
    if (p->x < q->x) return 1;
    return (p->idx < q->idx) ? -1 : (p->idx > q->idx);
}

/*
 * Probabilities of one logit row, "full probability distributions" of
 * §Target-Draft: p = softmax(x / T), then the top-p nucleus when
 * top_p < 1, renormalised.  T must be > 0 here.
 *
 * topp_margin (may be NULL) receives the distance, in probability mass,
 * between top_p and the nearest "mass before this token" value among the
 * last kept and the first dropped token (+inf when top-p is off).
 * Returns ORC_OK or ORC_ERR_NONFINITE.
 */
int orc_row_probs(const double* x, int V, double T, double top_p, double* p, double* topp_margin)
{
    if (topp_margin) *topp_margin = INFINITY;
    if (!row_valid(x, V)) return ORC_ERR_NONFINITE;
    double m = -INFINITY;
    for (int v = 0; v < V; ++v)
        if (x[v] > m) m = x[v];
    double Z = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = isinf(x[v]) ? 0.0 : exp((x[v] - m) / T);
        Z += p[v];
    }
    for (int v = 0; v < V; ++v) p[v] /= Z;
    if (!(top_p < 1.0)) return ORC_OK;

    keyed* order = (keyed*)malloc(sizeof(keyed) * (size_t)V);
    for (int v = 0; v < V; ++v) { order[v].x = x[v]; order[v].idx = v; }
    qsort(order, (size_t)V, sizeof(keyed), keyed_cmp);
    unsigned char* keep = (unsigned char*)calloc((size_t)V, 1);
    double before = 0.0, last_kept = -INFINITY, first_dropped = INFINITY;
    for (int r = 0; r < V; ++r) {
        int v = order[r].idx;
        if (before < top_p) {
            keep[v] = 1;
            last_kept = before;
        } else if (first_dropped == INFINITY) {
            first_dropped = before;
        }
        before += p[v];
    }
    if (topp_margin) {
        double a = top_p - last_kept, b = first_dropped - top_p;
        *topp_margin = a < b ? a : b;
    }
    double ZN = 0.0;
    for (int v = 0; v < V; ++v)
        if (keep[v]) ZN += p[v];
    for (int v = 0; v < V; ++v) p[v] = keep[v] ? p[v] / ZN : 0.0;
    free(keep);
    free(order);
    return ORC_OK;
}

/*
 * Inverse-CDF draw from non-negative weights w (index order): the smallest
 * v with C(v) > u * C(V-1), C the inclusive running sum.  Returns -1 when
 * C(V-1) == 0.  margin (may be NULL) receives the distance from u*C(V-1) to
 * the nearer edge of the chosen token's interval, divided by C(V-1).
 */
int orc_sample_inverse_cdf(const double* w, int V, double u, double* margin)
{
    double total = 0.0;
    for (int v = 0; v < V; ++v) total += w[v];
    if (margin) *margin = INFINITY;
    if (!(total > 0.0)) return -1;
    double target = u * total, c = 0.0;
    for (int v = 0; v < V; ++v) {
        double prev = c;
        c += w[v];
        if (c > target) {
            if (margin) {
                double a = (target - prev) / total, b = (c - target) / total;
                *margin = a < b ? a : b;
            }
            return v;
        }
    }
    /* u < 1 makes this unreachable up to rounding; take the last positive. */
    for (int v = V - 1; v >= 0; --v)
        if (w[v] > 0.0) { if (margin) *margin = 0.0; return v; }
    return -1;
}

static void min_into(double* m, double x)
{
    if (x < *m) *m = x;
}

/* Optional record of what a single-request verification did, for the
 * brute-force enumerator in tests: the threshold each accept test compared
 * u against, its outcome, and the weights of the final draw. */
typedef struct {
    int n_dec;
    double ratio[256];
    int accepted[256];
    int final_kind;   /* 0 residual / all children rejected, 1 bonus, 2 greedy, 3 invalid */
    double* final_w;  /* caller buffer [V] or NULL */
} orc_trace;

/* ------------------------------------------------------------------ */
/* Linear verification of one request (§Speculative decoding,         */
/* §Target-Draft).                                                     */
/* ------------------------------------------------------------------ */
/*
 * tgt: (k+1) rows of V target logits; row i scores the token after the
 *      prefix plus d_1..d_i.
 * drf: k rows of V draft logits; row i is the distribution d_{i+1} was drawn
 *      from (unused when T == 0, may be NULL then).
 * d:   k drafted tokens d_1..d_k.
 * u_acc[i]: uniform for the accept test of d_{i+1};
 * u_res[i]: uniform for the residual draw when d_{i+1} is the first reject;
 * u_bon:    uniform for the bonus draw after a full accept.
 * Outputs: *a_out accepted count, tokens[k+1] (d_1..d_a, t*, then -1),
 *          acc_prob[k] = min(1, p/q) per drafted token (may be NULL),
 *          tok_p[2k] = (p_i(d_{i+1}), q_i(d_{i+1})) pairs (may be NULL),
 *          *margin the smallest decision margin met (may be NULL).
 * Returns ORC_OK or an ORC_ERR_* bit for an invalid request, in which case
 * the outputs hold the fallback (a = 0, t* = argmax of target row 0).
 */
int orc_linear_request(const double* tgt, const double* drf, const int32_t* d, int k, int V,
                       double T, double top_p, const double* u_acc, const double* u_res, double u_bon,
                       int32_t* a_out, int32_t* tokens, double* acc_prob, double* tok_p,
                       double* margin, orc_trace* tr)
{
    double mg = INFINITY;
    int status = ORC_OK;
    for (int i = 0; i < k + 1; ++i) tokens[i] = -1;
    for (int i = 0; i < k; ++i) {
        if (acc_prob) acc_prob[i] = 0.0;
        if (tok_p) { tok_p[2 * i] = 0.0; tok_p[2 * i + 1] = 0.0; }
    }
    if (tr) { tr->n_dec = 0; tr->final_kind = 3; }
    for (int i = 0; i < k; ++i)
        if (d[i] < 0 || d[i] >= V) status |= ORC_ERR_TOKEN;

    if (T == 0.0) {
        int* g = (int*)malloc(sizeof(int) * (size_t)(k + 1));
        for (int i = 0; i <= k && !status; ++i) {
            if (!row_valid(tgt + (size_t)i * V, V)) status |= ORC_ERR_NONFINITE;
            g[i] = orc_argmax(tgt + (size_t)i * V, V);
        }
        if (!status) {
            int a = 0;
            while (a < k && d[a] == g[a]) ++a;
            for (int i = 0; i < k; ++i) {
                if (acc_prob) acc_prob[i] = (d[i] == g[i]) ? 1.0 : 0.0;
                if (tok_p) { tok_p[2 * i] = (d[i] == g[i]) ? 1.0 : 0.0; tok_p[2 * i + 1] = 1.0; }
            }
            for (int i = 0; i < a; ++i) tokens[i] = d[i];
            tokens[a] = g[a];
            *a_out = a;
            if (tr) tr->final_kind = 2;
        }
        free(g);
    } else {
        double* P = (double*)malloc(sizeof(double) * (size_t)(k + 1) * V);
        double* Q = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * V);
        double* tm = (double*)malloc(sizeof(double) * (size_t)(2 * k + 1));
        for (int i = 0; i <= k; ++i)
            status |= orc_row_probs(tgt + (size_t)i * V, V, T, top_p, P + (size_t)i * V, &tm[i]);
        for (int i = 0; i < k; ++i)
            status |= orc_row_probs(drf + (size_t)i * V, V, T, top_p, Q + (size_t)i * V, &tm[k + 1 + i]);
        if (!status) {
            double* ratio = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
            for (int i = 0; i < k; ++i) {
                double p = P[(size_t)i * V + d[i]], q = Q[(size_t)i * V + d[i]];
                ratio[i] = q > 0.0 ? p / q : 0.0;
                if (acc_prob) acc_prob[i] = ratio[i] < 1.0 ? ratio[i] : 1.0;
                if (tok_p) { tok_p[2 * i] = p; tok_p[2 * i + 1] = q; }
            }
            int a = 0;
            while (a < k) {
                min_into(&mg, fabs(u_acc[a] - ratio[a]));
                min_into(&mg, tm[a]);
                min_into(&mg, tm[k + 1 + a]);
                int acc = u_acc[a] < ratio[a];
                if (tr && tr->n_dec < 256) { tr->ratio[tr->n_dec] = ratio[a]; tr->accepted[tr->n_dec] = acc; tr->n_dec++; }
                if (!acc) break;
                ++a;
            }
            min_into(&mg, tm[a]);
            double* w = (double*)malloc(sizeof(double) * (size_t)V);
            const double* Pa = P + (size_t)a * V;
            int t;
            double sm;
            if (a < k) {
                const double* Qa = Q + (size_t)a * V;
                for (int v = 0; v < V; ++v) { double r = Pa[v] - Qa[v]; w[v] = r > 0.0 ? r : 0.0; }
                t = orc_sample_inverse_cdf(w, V, u_res[a], &sm);
                if (t < 0) {
                    memcpy(w, Pa, sizeof(double) * (size_t)V);
                    t = orc_sample_inverse_cdf(w, V, u_res[a], &sm);
                }
                if (tr) tr->final_kind = 0;
            } else {
                memcpy(w, Pa, sizeof(double) * (size_t)V);
                t = orc_sample_inverse_cdf(w, V, u_bon, &sm);
                if (tr) tr->final_kind = 1;
            }
            min_into(&mg, sm);
            if (tr && tr->final_w) memcpy(tr->final_w, w, sizeof(double) * (size_t)V);
            for (int i = 0; i < a; ++i) tokens[i] = d[i];
            tokens[a] = t;
            *a_out = a;
            free(w);
            free(ratio);
        }
        free(tm);
        free(Q);
        free(P);
    }
    if (status) {
        for (int i = 0; i < k + 1; ++i) tokens[i] = -1;
        for (int i = 0; i < k; ++i) {
            if (acc_prob) acc_prob[i] = 0.0;
            if (tok_p) { tok_p[2 * i] = 0.0; tok_p[2 * i + 1] = 0.0; }
        }
        tokens[0] = orc_argmax(tgt, V);
        *a_out = 0;
        mg = INFINITY;
        if (tr) tr->final_kind = 3;
    }
    if (margin) *margin = mg;
    return status;
}

/* Batched linear verification with Philox uniforms; positions of drafted
 * token i (1-based) are positions[b] + i. */
int orc_verify_linear(const double* tgt, const double* drf, const int32_t* drafts, int B, int k, int V,
                      const int64_t* req_ids, const int64_t* positions, double T, double top_p, uint64_t seed,
                      int32_t* accepted_len, int32_t* out_tokens, double* accept_prob, double* tok_p,
                      int32_t* len_hist, double* margins, int32_t* dev_error)
{
    int err = 0;
    double* u_acc = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    double* u_res = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    if (len_hist)
        for (int i = 0; i <= k; ++i) len_hist[i] = 0;
    for (int b = 0; b < B; ++b) {
        int64_t rq = req_ids ? req_ids[b] : b;
        int64_t base = positions ? positions[b] : 0;
        for (int i = 0; i < k; ++i) {
            u_acc[i] = orc_uniform(seed, rq, base + i + 1, ORC_PURPOSE_ACCEPT, 0);
            u_res[i] = orc_uniform(seed, rq, base + i + 1, ORC_PURPOSE_RESIDUAL, 0);
        }
        double u_bon = orc_uniform(seed, rq, base + k + 1, ORC_PURPOSE_BONUS, 0);
        int32_t a = 0;
        err |= orc_linear_request(tgt + (size_t)b * (k + 1) * V, drf ? drf + (size_t)b * k * V : NULL,
                                  drafts + (size_t)b * k, k, V, T, top_p, u_acc, u_res, u_bon, &a,
                                  out_tokens + (size_t)b * (k + 1), accept_prob ? accept_prob + (size_t)b * k : NULL,
                                  tok_p ? tok_p + (size_t)b * 2 * k : NULL, margins ? margins + b : NULL, NULL);
        accepted_len[b] = a;
        if (len_hist) len_hist[a] += 1;
    }
    free(u_res);
    free(u_acc);
    if (dev_error) *dev_error = err;
    return err;
}

/* ------------------------------------------------------------------ */
/* Tree verification of one request (§EAGLE).                         */
/* ------------------------------------------------------------------ */

/* Depth of every node; returns -1 when parent[] is not a topologically
 * ordered tree rooted at node 0 (parent[0] == -1, 0 <= parent[i] < i). */
int orc_tree_depths(const int32_t* parent, int N, int32_t* depth)
{
    if (N < 1 || parent[0] != -1) return -1;
    depth[0] = 0;
    int dmax = 0;
    for (int i = 1; i < N; ++i) {
        if (parent[i] < 0 || parent[i] >= i) return -1;
        depth[i] = depth[parent[i]] + 1;
        if (depth[i] > dmax) dmax = depth[i];
    }
    return dmax;
}

/*
 * tgt, drf: N rows of V logits; row n scores the token after node n's path.
 * tok[n]: the token of node n (tok[0] unused).  Children of n are the nodes
 * i with parent[i] == n, tested in increasing index order.
 * u_acc[depth * Kmax + j]: uniform of the test of the j-th child at that
 * depth; u_res[depth], u_bon[depth]: uniform of the final draw there.
 * mode: ORC_CHILD_WOR (children drawn from q without replacement),
 *       ORC_CHILD_IID (with replacement), ORC_CHILD_DET (top-K of q).
 * Outputs: *a_out accepted depth, path[Dmax+1] (0, accepted nodes, -1 pad),
 *          tokens[Dmax+1] (accepted tokens, t*, -1 pad).
 */
int orc_tree_request(const double* tgt, const double* drf, const int32_t* tok, const int32_t* parent,
                     int N, int V, double T, double top_p, int mode,
                     const double* u_acc, int Kmax, const double* u_res, const double* u_bon,
                     int32_t* a_out, int32_t* path, int32_t* tokens, double* margin, orc_trace* tr)
{
    int32_t* depth = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    int dmax = orc_tree_depths(parent, N, depth);
    int status = ORC_OK;
    double mg = INFINITY;
    int W = (dmax < 0 ? 0 : dmax) + 1;
    for (int i = 0; i < W; ++i) { path[i] = -1; tokens[i] = -1; }
    if (tr) { tr->n_dec = 0; tr->final_kind = 3; }
    if (dmax < 0) status |= ORC_ERR_PARENT;
    for (int i = 1; i < N && !status; ++i)
        if (tok[i] < 0 || tok[i] >= V) status |= ORC_ERR_TOKEN;

    int* ch = (int*)malloc(sizeof(int) * (size_t)N);
    double* P = (double*)malloc(sizeof(double) * (size_t)V);
    double* Q = (double*)malloc(sizeof(double) * (size_t)V);
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    int n = 0, dep = 0, t = -1;
    if (!status) path[0] = 0;
    while (!status) {
        int m = 0;
        for (int i = n + 1; i < N; ++i)
            if (parent[i] == n) ch[m++] = i;
        const double* xp = tgt + (size_t)n * V;
        if (T == 0.0) {
            if (!row_valid(xp, V)) { status |= ORC_ERR_NONFINITE; break; }
            int g = orc_argmax(xp, V), next = -1;
            for (int j = 0; j < m; ++j)
                if (tok[ch[j]] == g) { next = ch[j]; break; }
            if (next < 0) { t = g; if (tr) tr->final_kind = 2; break; }
            ++dep; path[dep] = next; tokens[dep - 1] = tok[next]; n = next;
            continue;
        }
        double tmp;
        status |= orc_row_probs(xp, V, T, top_p, P, &tmp);
        if (status) break;
        min_into(&mg, tmp);
        if (m == 0) {
            double sm;
            memcpy(w, P, sizeof(double) * (size_t)V);
            t = orc_sample_inverse_cdf(w, V, u_bon[dep], &sm);
            min_into(&mg, sm);
            if (tr) { tr->final_kind = 1; if (tr->final_w) memcpy(tr->final_w, w, sizeof(double) * (size_t)V); }
            break;
        }
        if (mode != ORC_CHILD_DET) {
            status |= orc_row_probs(drf + (size_t)n * V, V, T, top_p, Q, &tmp);
            if (status) break;
            min_into(&mg, tmp);
        }
        int next = -1;
        for (int j = 0; j < m; ++j) {
            int x = tok[ch[j]];
            double ratio;
            if (mode == ORC_CHILD_DET) ratio = P[x];
            else ratio = Q[x] > 0.0 ? P[x] / Q[x] : 0.0;
            double u = u_acc[(size_t)dep * Kmax + j];
            min_into(&mg, fabs(u - ratio));
            int acc = u < ratio;
            if (tr && tr->n_dec < 256) { tr->ratio[tr->n_dec] = ratio; tr->accepted[tr->n_dec] = acc; tr->n_dec++; }
            if (acc) { next = ch[j]; break; }
            if (mode == ORC_CHILD_DET) {
                double s = 0.0;
                P[x] = 0.0;
                for (int v = 0; v < V; ++v) s += P[v];
                if (s > 0.0)
                    for (int v = 0; v < V; ++v) P[v] /= s;
            } else {
                double s = 0.0;
                for (int v = 0; v < V; ++v) { double r = P[v] - Q[v]; w[v] = r > 0.0 ? r : 0.0; s += w[v]; }
                if (s > 0.0)
                    for (int v = 0; v < V; ++v) P[v] = w[v] / s;
                if (mode == ORC_CHILD_WOR) {
                    double sq = 0.0;
                    Q[x] = 0.0;
                    for (int v = 0; v < V; ++v) sq += Q[v];
                    if (sq > 0.0)
                        for (int v = 0; v < V; ++v) Q[v] /= sq;
                }
            }
        }
        if (next >= 0) {
            ++dep; path[dep] = next; tokens[dep - 1] = tok[next]; n = next;
            continue;
        }
        double sm;
        memcpy(w, P, sizeof(double) * (size_t)V);
        t = orc_sample_inverse_cdf(w, V, u_res[dep], &sm);
        min_into(&mg, sm);
        if (tr) { tr->final_kind = 0; if (tr->final_w) memcpy(tr->final_w, w, sizeof(double) * (size_t)V); }
        break;
    }
    if (status) {
        for (int i = 0; i < W; ++i) { path[i] = -1; tokens[i] = -1; }
        path[0] = 0;
        tokens[0] = orc_argmax(tgt, V);
        *a_out = 0;
        mg = INFINITY;
        if (tr) tr->final_kind = 3;
    } else {
        tokens[dep] = t;
        *a_out = dep;
    }
    if (margin) *margin = mg;
    free(w);
    free(Q);
    free(P);
    free(ch);
    free(depth);
    return status;
}

/* Batched tree verification with Philox uniforms.  The decision at a node
 * of depth d uses position positions[b] + d + 1; child j uses round j. */
int orc_verify_tree(const double* tgt, const double* drf, const int32_t* node_tokens, const int32_t* parent,
                    int B, int N, int V, const int64_t* req_ids, const int64_t* positions,
                    double T, double top_p, uint64_t seed, int mode,
                    int32_t* accepted_len, int32_t* path_nodes, int32_t* out_tokens, double* margins,
                    int32_t* dev_error)
{
    int32_t* depth = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int dmax = orc_tree_depths(parent, N, depth);
    int W = (dmax < 0 ? 0 : dmax) + 1;
    int Kmax = N;
    double* u_acc = (double*)malloc(sizeof(double) * (size_t)W * Kmax);
    double* u_res = (double*)malloc(sizeof(double) * (size_t)W);
    double* u_bon = (double*)malloc(sizeof(double) * (size_t)W);
    int err = 0;
    for (int b = 0; b < B; ++b) {
        int64_t rq = req_ids ? req_ids[b] : b;
        int64_t base = positions ? positions[b] : 0;
        for (int dd = 0; dd < W; ++dd) {
            for (int j = 0; j < Kmax; ++j)
                u_acc[(size_t)dd * Kmax + j] = orc_uniform(seed, rq, base + dd + 1, ORC_PURPOSE_ACCEPT, j);
            u_res[dd] = orc_uniform(seed, rq, base + dd + 1, ORC_PURPOSE_RESIDUAL, 0);
            u_bon[dd] = orc_uniform(seed, rq, base + dd + 1, ORC_PURPOSE_BONUS, 0);
        }
        int32_t a = 0;
        err |= orc_tree_request(tgt + (size_t)b * N * V, drf ? drf + (size_t)b * N * V : NULL,
                                node_tokens + (size_t)b * N, parent, N, V, T, top_p, mode,
                                u_acc, Kmax, u_res, u_bon, &a, path_nodes + (size_t)b * W,
                                out_tokens + (size_t)b * W, margins ? margins + b : NULL, NULL);
        accepted_len[b] = a;
    }
    free(u_bon);
    free(u_res);
    free(u_acc);
    free(depth);
    if (dev_error) *dev_error = err;
    return err;
}

/* ------------------------------------------------------------------ */
/* Compaction (§MTP: t_{i+1} pairs with H_i; §MTP schedule for a      */
/* single token: a kernel inserts the next tokens into their slots).  */
/* ------------------------------------------------------------------ */
/*
 * hidden: [B, T, H] rows (any 2-byte element type, copied bit for bit).
 * For request b with a_b accepted tokens, rows r = 0..a_b of the output
 * block starting at offsets[b] receive hidden[b, src_r, :] with
 * src_r = path_nodes[b, r] (or r when path_nodes is NULL) and
 * next_tokens[offsets[b] + r] = out_tokens[b, r].  offsets[b+1] =
 * offsets[b] + a_b + 1.  A request whose a_b is outside [0, W-1], or whose
 * source row is outside [0, T), contributes no rows and sets an error bit.
 */
int orc_compact(const uint16_t* hidden, int B, int T, int H, const int32_t* accepted_len,
                const int32_t* path_nodes, const int32_t* out_tokens, int W,
                uint16_t* out_hidden, int32_t* offsets, int32_t* next_tokens, int32_t* dev_error)
{
    int err = 0;
    offsets[0] = 0;
    for (int b = 0; b < B; ++b) {
        int a = accepted_len[b];
        int ok = a >= 0 && a < W;
        for (int r = 0; ok && r <= a; ++r) {
            int src = path_nodes ? path_nodes[(size_t)b * W + r] : r;
            if (src < 0 || src >= T) ok = 0;
        }
        if (!ok) { err |= ORC_ERR_LENGTH; offsets[b + 1] = offsets[b]; continue; }
        for (int r = 0; r <= a; ++r) {
            int src = path_nodes ? path_nodes[(size_t)b * W + r] : r;
            int dst = offsets[b] + r;
            memcpy(out_hidden + (size_t)dst * H, hidden + ((size_t)b * T + src) * H, sizeof(uint16_t) * (size_t)H);
            next_tokens[dst] = out_tokens[(size_t)b * W + r];
        }
        offsets[b + 1] = offsets[b] + a + 1;
    }
    if (dev_error) *dev_error = err;
    return err;
}

/* ------------------------------------------------------------------ */
/* Draft-side draws used by the test harness to make draft tokens.    */
/* ------------------------------------------------------------------ */

/* One token per row from filter(softmax(x / T)); T == 0 takes the argmax.
 * Row r uses Philox(seed, req[r], pos[r], DRAFT, 0). */
int orc_sample_rows(const double* x, int R, int V, double T, double top_p, uint64_t seed,
                    const int64_t* req, const int64_t* pos, int32_t* out)
{
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    int err = 0;
    for (int r = 0; r < R; ++r) {
        const double* row = x + (size_t)r * V;
        if (T == 0.0) { out[r] = orc_argmax(row, V); continue; }
        if (orc_row_probs(row, V, T, top_p, p, NULL) != ORC_OK) { err |= ORC_ERR_NONFINITE; out[r] = orc_argmax(row, V); continue; }
        double u = orc_uniform(seed, req[r], pos[r], ORC_PURPOSE_DRAFT, 0);
        out[r] = orc_sample_inverse_cdf(p, V, u, NULL);
    }
    free(p);
    return err;
}

/* K children tokens of one node drawn from filter(softmax(x / T)):
 * WOR draws without replacement (each draw renormalises the rest), IID with
 * replacement, DET takes the K highest-probability tokens (logit desc,
 * index asc).  Draw j uses Philox(seed, req, pos, DRAFT, j). */
int orc_draw_children(const double* x, int V, double T, double top_p, int K, int mode, uint64_t seed,
                      int64_t req, int64_t pos, int32_t* out)
{
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    int err = orc_row_probs(x, V, T > 0.0 ? T : 1.0, top_p, p, NULL);
    if (err == ORC_OK) {
        if (mode == ORC_CHILD_DET) {
            keyed* order = (keyed*)malloc(sizeof(keyed) * (size_t)V);
            for (int v = 0; v < V; ++v) { order[v].x = x[v]; order[v].idx = v; }
            qsort(order, (size_t)V, sizeof(keyed), keyed_cmp);
            for (int j = 0; j < K; ++j) out[j] = order[j < V ? j : V - 1].idx;
            free(order);
        } else {
            for (int j = 0; j < K; ++j) {
                double u = orc_uniform(seed, req, pos, ORC_PURPOSE_DRAFT, j);
                int t = orc_sample_inverse_cdf(p, V, u, NULL);
                out[j] = t;
                if (mode == ORC_CHILD_WOR && t >= 0) p[t] = 0.0;
            }
        }
    }
    free(p);
    return err;
}
