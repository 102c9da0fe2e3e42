/*
 * oracle.c -- plain float64 CPU oracle for speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package entry's smoke check and the
 * benchmark's CPU-baseline leg may load or call this file. It shares no code, header,
 * table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes (sources are the web pages on tree speculation; citations name the page
 * and the section):
 *   - EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and lossless throughput",
 *     commit 4b728e2 "grammar-trie tree speculation with exact acceptance": a trie of N draft
 *     nodes is verified in one tree-attention forward; greedy decoding keeps the argmax path;
 *     sampling uses standard (SpecInfer-style) rejection sampling against the draft, so the
 *     output distribution equals the target's.
 *   - IluvatarLabs/vllm PR #3 "SCV vectorized masking": an acceptance mask per request built
 *     from the draft (here: the ancestor mask of the tree).
 * Where the pages are silent the plainest reading is taken; each reading is marked READING.
 *
 * Every quantity is computed in float64 from the exact input values (bf16 and fp32 are
 * widened exactly). Loops run in plain index order; there is no blocking or fusion.
 *
 * Parity pins: tests/test_oracle_*.py (hand-worked goldens, brute-force enumeration of the
 * output distribution against target autoregressive sampling, Monte-Carlo chi-square,
 * invariants, closed forms, planted-mistake checks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_DRAFT_POINT = 0, OR_DRAFT_PROBS_F32 = 1, OR_DRAFT_LOGITS = 2 };
enum { OR_OK = 0, OR_BAD_PARENT = 1, OR_BAD_TOKEN = 2, OR_BAD_ROW = 3, OR_BAD_UNIFORM = 4 };

/* ---- input decoding ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double elem(const void *base, int dtype, int64_t i) {
    if (dtype == OR_F32) return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static size_t elem_size(int dtype) { return dtype == OR_F32 ? 4 : 2; }

static const void *row_ptr(const void *base, int dtype, int64_t row, int64_t V) {
    return (const char *)base + (size_t)row * (size_t)V * elem_size(dtype);
}

/* ---- tree ----------------------------------------------------------------------------- */

/* READING: parent[0] == -1 and 0 <= parent[i] < i (topological order) for i > 0. */
static int tree_valid(const int32_t *parent, int N) {
    if (N < 1 || parent[0] != -1) return 0;
    for (int i = 1; i < N; i++)
        if (parent[i] < 0 || parent[i] >= i) return 0;
    return 1;
}

/* Ancestor mask and depth by walking each node's parent chain to the root. Query i may
 * attend to key j iff bit j of anc[i] is set (self included). */
int oracle_build_mask(const int32_t *parent, int B, int N, uint64_t *anc, int32_t *depth,
                      int32_t *status) {
    if (N < 1 || N > 64 || B < 0) return -1;
    for (int b = 0; b < B; b++) {
        const int32_t *par = parent + (size_t)b * N;
        if (!tree_valid(par, N)) {
            status[b] = OR_BAD_PARENT;
            for (int i = 0; i < N; i++) {
                anc[(size_t)b * N + i] = 0;
                depth[(size_t)b * N + i] = -1;
            }
            continue;
        }
        status[b] = OR_OK;
        for (int i = 0; i < N; i++) {
            uint64_t m = 0;
            int d = -1;
            for (int j = i; j != -1; j = par[j]) {
                m |= (uint64_t)1 << j;
                d++;
            }
            anc[(size_t)b * N + i] = m;
            depth[(size_t)b * N + i] = d;
        }
    }
    return 0;
}

/* ---- rows ------------------------------------------------------------------------------- */

/* READING: a row the walk needs is unusable if it holds a NaN or +inf, or every entry is
 * -inf. -inf entries alone are allowed and carry zero probability. */
static int row_bad(const void *row, int dtype, int64_t V) {
    int any_finite_or_neg = 0;
    for (int64_t v = 0; v < V; v++) {
        double z = elem(row, dtype, v);
        if (isnan(z) || z == INFINITY) return 1;
        if (z != -INFINITY) any_finite_or_neg = 1;
    }
    return !any_finite_or_neg;
}

/* Lowest index v maximising z[v]. */
static int64_t row_argmax(const void *row, int dtype, int64_t V) {
    int64_t a = 0;
    double best = elem(row, dtype, 0);
    for (int64_t v = 1; v < V; v++) {
        double z = elem(row, dtype, v);
        if (z > best) {
            best = z;
            a = v;
        }
    }
    return a;
}

/* p = softmax(z / T), formed as exp((z - m)/T) / sum_w exp((z_w - m)/T) with m = max z. */
static void row_softmax(const void *row, int dtype, int64_t V, double T, double *p) {
    double m = -INFINITY;
    for (int64_t v = 0; v < V; v++) {
        double z = elem(row, dtype, v);
        if (z > m) m = z;
    }
    double S = 0.0;
    for (int64_t v = 0; v < V; v++) {
        p[v] = exp((elem(row, dtype, v) - m) / T);
        S += p[v];
    }
    for (int64_t v = 0; v < V; v++) p[v] /= S;
}

/* Exported row statistics: max m, lowest-index argmax, S = sum_v exp((z_v - m)/T)
 * (T > 0; S is left 0 when T == 0), and the bad-row flag. */
int oracle_row_stats(const void *row, int dtype, int64_t V, double T, double *m_out,
                     double *S_out, int64_t *argmax_out, int32_t *bad_out) {
    if (V < 1) return -1;
    *bad_out = row_bad(row, dtype, V);
    *argmax_out = row_argmax(row, dtype, V);
    double m = -INFINITY;
    for (int64_t v = 0; v < V; v++) {
        double z = elem(row, dtype, v);
        if (z > m) m = z;
    }
    *m_out = m;
    double S = 0.0;
    if (T > 0)
        for (int64_t v = 0; v < V; v++) S += exp((elem(row, dtype, v) - m) / T);
    *S_out = S;
    return 0;
}

int oracle_row_softmax(const void *row, int dtype, int64_t V, double T, double *p) {
    if (V < 1 || !(T > 0)) return -1;
    row_softmax(row, dtype, V, T, p);
    return 0;
}

/* Half-width, relative to S, of the window of draws reported beside every inverse CDF: the
 * tolerance below which the comparisons accept a different token from an arithmetic that
 * rounds the running sums differently. */
#define OR_CDF_WINDOW 1e-6

/* InvCDF(r, u): with S = sum r and tau = u*S, the smallest v whose running sum exceeds
 * tau; if rounding leaves none, the largest v with r[v] > 0. The margin is the distance of
 * tau to the nearer end of the chosen interval, over S (0 on the fallback). *alt is the token
 * with r > 0 on the other side of that nearer end (v itself if there is none): the draw an
 * arithmetic that rounds the running sums differently may make when the margin is tiny.
 * win[0..1] is the first and last token with r > 0 whose interval [C(v) - r(v), C(v))
 * comes within OR_CDF_WINDOW * S of tau: every token such an arithmetic can draw when its
 * tau and running sums are off by less than that (tokens of tiny mass can put several of
 * them inside the window). */
static void cdf_window(const double *r, int64_t V, double S, double tau, int64_t drawn,
                       int64_t *win) {
    double delta = OR_CDF_WINDOW * S, C = 0.0;
    win[0] = -1;
    win[1] = -1;
    for (int64_t v = 0; v < V; v++) {
        double Cprev = C;
        C += r[v];
        if (!(r[v] > 0.0)) continue;
        if (Cprev >= tau + delta) break;
        if (win[0] < 0 && C > tau - delta) win[0] = v;
        win[1] = v;
    }
    if (win[0] < 0 || win[0] > drawn) win[0] = drawn;
    if (win[1] < drawn) win[1] = drawn;
}

static int64_t inv_cdf(const double *r, int64_t V, double u, double *margin, int64_t *alt,
                       int64_t *win) {
    double S = 0.0;
    for (int64_t v = 0; v < V; v++) S += r[v];
    double tau = u * S;
    double C = 0.0;
    for (int64_t v = 0; v < V; v++) {
        double Cprev = C;
        C += r[v];
        if (C > tau) {
            double a = C - tau, b = tau - Cprev;
            *margin = (a < b ? a : b) / S;
            *alt = v;
            if (a < b) {
                for (int64_t w = v + 1; w < V; w++)
                    if (r[w] > 0) {
                        *alt = w;
                        break;
                    }
            } else {
                for (int64_t w = v - 1; w >= 0; w--)
                    if (r[w] > 0) {
                        *alt = w;
                        break;
                    }
            }
            cdf_window(r, V, S, tau, v, win);
            return v;
        }
    }
    *margin = 0.0;
    for (int64_t v = V - 1; v >= 0; v--)
        if (r[v] > 0) {
            *alt = v;
            cdf_window(r, V, S, tau, v, win);
            return v;
        }
    *alt = V - 1;
    win[0] = win[1] = V - 1;
    return V - 1;
}

int64_t oracle_inv_cdf(const double *r, int64_t V, double u, double *margin, int64_t *win) {
    int64_t alt;
    return inv_cdf(r, V, u, margin, &alt, win);
}

/* ---- per-request outputs ------------------------------------------------------------------ */

typedef struct {
    int32_t *accept_len, *out_tokens, *kv_commit, *bonus, *status;
} outputs;

static void write_failed(outputs o, int b, int N, int32_t code) {
    o.accept_len[b] = 0;
    o.bonus[b] = -1;
    o.status[b] = code;
    for (int i = 0; i < N; i++) {
        o.out_tokens[(size_t)b * N + i] = -1;
        o.kv_commit[(size_t)b * N + i] = -1;
    }
}

/* accept_len = L accepted non-root nodes; out_tokens = tokens of the accepted nodes in path
 * order then the bonus; kv_commit = root (0) then the accepted node ids; -1 padded.
 * READING: the root's KV is produced by the same verify forward and is committed too. */
static void write_path(outputs o, int b, int N, const int32_t *tok, const int *path, int L,
                       int32_t bonus) {
    o.accept_len[b] = L;
    o.bonus[b] = bonus;
    o.status[b] = OR_OK;
    for (int i = 0; i < N; i++) {
        o.out_tokens[(size_t)b * N + i] = -1;
        o.kv_commit[(size_t)b * N + i] = -1;
    }
    o.kv_commit[(size_t)b * N + 0] = 0;
    for (int j = 0; j < L; j++) {
        o.out_tokens[(size_t)b * N + j] = tok[path[j]];
        o.kv_commit[(size_t)b * N + j + 1] = path[j];
    }
    o.out_tokens[(size_t)b * N + L] = bonus;
}

/* Shared request validation: structure first, then draft tokens of non-root nodes
 * (the root's token is ignored). */
static int32_t check_request(const int32_t *par, const int32_t *tok, int N, int64_t V) {
    if (!tree_valid(par, N)) return OR_BAD_PARENT;
    for (int i = 1; i < N; i++)
        if (tok[i] < 0 || tok[i] >= V) return OR_BAD_TOKEN;
    return OR_OK;
}

/* ---- greedy ------------------------------------------------------------------------------- */

/* Greedy: starting at the root, find a = argmax of the current node's row (lowest index on
 * ties); move to the first child in trie order (ascending node index) whose draft token
 * equals a; stop when none does. The bonus is a at the stop node.
 * READING: siblings are ordered by node index; with duplicate sibling tokens the first
 * one in that order is taken. */
static void greedy_one(const void *logits, int dtype, int b, int N, int64_t V,
                       const int32_t *tok, const int32_t *par, outputs o) {
    int32_t st = check_request(par, tok, N, V);
    if (st != OR_OK) {
        write_failed(o, b, N, st);
        return;
    }
    int path[64];
    int L = 0, node = 0;
    int64_t a;
    for (;;) {
        const void *row = row_ptr(logits, dtype, (int64_t)b * N + node, V);
        if (row_bad(row, dtype, V)) {
            write_failed(o, b, N, OR_BAD_ROW);
            return;
        }
        a = row_argmax(row, dtype, V);
        int next = -1;
        for (int c = node + 1; c < N; c++)
            if (par[c] == node && tok[c] == a) {
                next = c;
                break;
            }
        if (next < 0) break;
        path[L++] = next;
        node = next;
    }
    write_path(o, b, N, tok, path, L, (int32_t)a);
}

int oracle_verify_greedy(const void *logits, int dtype, int B, int N, int64_t V,
                         const int32_t *draft_token, const int32_t *parent,
                         int32_t *accept_len, int32_t *out_tokens, int32_t *kv_commit,
                         int32_t *bonus, int32_t *status, int nthreads) {
    if (B < 0 || N < 1 || N > 64 || V < 1 || (dtype != OR_F32 && dtype != OR_BF16)) return -1;
    outputs o = {accept_len, out_tokens, kv_commit, bonus, status};
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int b = 0; b < B; b++)
        greedy_one(logits, dtype, b, N, V, draft_token + (size_t)b * N,
                   parent + (size_t)b * N, o);
    return 0;
}

/* ---- sampling ------------------------------------------------------------------------------- */

typedef struct {
    double *p, *r, *q, *tmp;
} scratch;

/* Point-mass drafts (a deterministic trie: the draft puts probability 1 on each drafted
 * child's token). At the current node with target p and rejected set R (tokens already
 * rejected at this node), child c with token t is accepted iff u[c] < rhat with
 *     rhat = p(t) / sum_{v not in R} p(v)   (0 if t is in R),
 * i.e. min(1, r(t)/q(t)) with q(t) = 1 and r the residual norm(max(p - q, 0)) after the
 * earlier siblings' point masses were removed. On rejection t joins R. When no child is
 * accepted (or the node is a leaf) the bonus is InvCDF(p with R zeroed, u[N]).
 * READING: u[b][c] is consumed when child c is tested, u[b][N] draws the bonus, u[b][0] is
 * unused; the test is strict (u < rhat). */
static int32_t sample_point(const void *logits, int dtype, int b, int N, int64_t V, double T,
                            const int32_t *tok, const int32_t *par, const float *u,
                            scratch s, int *path, int *L_out, double *dmargin, double *cmargin,
                            int32_t *calt, int32_t *cwin) {
    int node = 0, L = 0;
    double *p = s.p, *r = s.r;
    char *inR = (char *)s.tmp; /* V bytes */
    for (;;) {
        const void *row = row_ptr(logits, dtype, (int64_t)b * N + node, V);
        if (row_bad(row, dtype, V)) return -OR_BAD_ROW;
        row_softmax(row, dtype, V, T, p);
        memset(inR, 0, (size_t)V);
        int next = -1;
        for (int c = node + 1; c < N && next < 0; c++) {
            if (par[c] != node) continue;
            int32_t t = tok[c];
            double rhat = 0.0;
            if (!inR[t]) {
                double S = 0.0;
                for (int64_t v = 0; v < V; v++)
                    if (!inR[v]) S += p[v];
                rhat = p[t] / S;
            }
            double uc = (double)u[c];
            double mg = fabs(uc - rhat);
            if (mg < *dmargin) *dmargin = mg;
            if (uc < rhat)
                next = c;
            else
                inR[t] = 1;
        }
        if (next < 0) break;
        path[L++] = next;
        node = next;
    }
    for (int64_t v = 0; v < V; v++) r[v] = inR[v] ? 0.0 : p[v];
    double cm;
    int64_t alt, win[2];
    int64_t bonus = inv_cdf(r, V, (double)u[N], &cm, &alt, win);
    *cmargin = cm;
    *calt = (int32_t)alt;
    cwin[0] = (int32_t)win[0];
    cwin[1] = (int32_t)win[1];
    *L_out = L;
    return (int32_t)bonus;
}

/* Draft row of node i: the distribution that drafted i's children. PROBS_F32 rows are used
 * as given; LOGITS rows are softmax(d / T) with the target's temperature (READING). */
static int draft_row(const void *draft, int draft_kind, int draft_dtype, int64_t row, int64_t V,
                     double T, double *q) {
    if (draft_kind == OR_DRAFT_PROBS_F32) {
        const float *pr = (const float *)draft + (size_t)row * V;
        for (int64_t v = 0; v < V; v++) {
            double x = pr[v];
            if (!(x >= 0.0) || isinf(x)) return 0;
            q[v] = x;
        }
        return 1;
    }
    const void *rw = row_ptr(draft, draft_dtype, row, V);
    if (row_bad(rw, draft_dtype, V)) return 0;
    row_softmax(rw, draft_dtype, V, T, q);
    return 1;
}

/* Dense drafts (standard speculative sampling; SpecInfer's multi-step form on trees). At
 * the current node the residual starts as r = p. Child c with token x, drafted from the
 * node's draft row q, is accepted iff u[c] * q(x) < r(x) (min(1, r(x)/q(x)) with a strict
 * test). On rejection r <- max(r - q, 0) / Z with Z = sum_v max(r(v) - q(v), 0); if Z == 0
 * (target and draft agree to rounding) the residual is kept unchanged and the case is
 * counted. When no child is accepted the bonus is InvCDF(r, u[N]); at a leaf r = p.
 * On a chain this is the standard rule: accept with min(1, p/q), on rejection sample
 * norm(max(p - q, 0)). */
static int32_t sample_dense(const void *logits, int dtype, int b, int N, int64_t V, double T,
                            const int32_t *tok, const int32_t *par, const void *draft,
                            int draft_kind, int draft_dtype, const float *u, scratch s,
                            int *path, int *L_out, double *dmargin, double *cmargin,
                            int32_t *degenerate, int32_t *calt, int32_t *cwin) {
    int node = 0, L = 0;
    double *p = s.p, *r = s.r, *q = s.q;
    for (;;) {
        int64_t grow = (int64_t)b * N + node;
        const void *row = row_ptr(logits, dtype, grow, V);
        if (row_bad(row, dtype, V)) return -OR_BAD_ROW;
        row_softmax(row, dtype, V, T, p);
        for (int64_t v = 0; v < V; v++) r[v] = p[v];
        int have_children = 0;
        for (int c = node + 1; c < N; c++)
            if (par[c] == node) have_children = 1;
        if (!have_children) break;
        if (!draft_row(draft, draft_kind, draft_dtype, grow, V, T, q)) return -OR_BAD_ROW;
        int next = -1;
        for (int c = node + 1; c < N && next < 0; c++) {
            if (par[c] != node) continue;
            int32_t x = tok[c];
            double lhs = (double)u[c] * q[x];
            /* decision margin in normalised terms: the test is u < r(x)/q(x) */
            double mg = q[x] > 0.0 ? fabs(lhs - r[x]) / q[x] : r[x];
            if (mg < *dmargin) *dmargin = mg;
            if (lhs < r[x]) {
                next = c;
                break;
            }
            double Z = 0.0;
            for (int64_t v = 0; v < V; v++) {
                double d = r[v] - q[v];
                Z += d > 0.0 ? d : 0.0;
            }
            if (Z == 0.0) {
                (*degenerate)++;
                continue;
            }
            for (int64_t v = 0; v < V; v++) {
                double d = r[v] - q[v];
                r[v] = (d > 0.0 ? d : 0.0) / Z;
            }
        }
        if (next < 0) break;
        path[L++] = next;
        node = next;
    }
    double cm;
    int64_t alt, win[2];
    int64_t bonus = inv_cdf(r, V, (double)u[N], &cm, &alt, win);
    *cmargin = cm;
    *calt = (int32_t)alt;
    cwin[0] = (int32_t)win[0];
    cwin[1] = (int32_t)win[1];
    *L_out = L;
    return (int32_t)bonus;
}

/* Sampling verify. T == 0 is greedy. Uniforms have shape [B, N+1]; every slot 1..N must lie
 * in [0, 1) or the request fails with status 4 (READING: checked before the walk, whether or
 * not the walk consumes the slot). decision_margin[b] is the smallest |u - r(x)/q(x)| over
 * the tests taken (= |u*q - r|/q, never below |u*q - r| as q <= 1; +inf if no test),
 * cdf_margin[b] the bonus draw's margin, cdf_alt[b] the token across the nearer boundary of
 * the drawn interval, cdf_window[b][0..1] the first and last token an arithmetic within
 * OR_CDF_WINDOW of tau can draw (see inv_cdf; -1 without a draw), degenerate[b] the number
 * of degenerate dense residuals. */
int oracle_verify_sample(const void *logits, int dtype, int B, int N, int64_t V,
                         const int32_t *draft_token, const int32_t *parent, const void *draft,
                         int draft_kind, int draft_dtype, double T, const float *uniforms,
                         int32_t *accept_len, int32_t *out_tokens, int32_t *kv_commit,
                         int32_t *bonus, int32_t *status, double *decision_margin,
                         double *cdf_margin, int32_t *cdf_alt, int32_t *cdf_window,
                         int32_t *degenerate, int nthreads) {
    if (B < 0 || N < 1 || N > 64 || V < 1 || (dtype != OR_F32 && dtype != OR_BF16)) return -1;
    if (!(T >= 0.0) || isinf(T)) return -1;
    if (draft_kind != OR_DRAFT_POINT && draft_kind != OR_DRAFT_PROBS_F32 &&
        draft_kind != OR_DRAFT_LOGITS)
        return -1;
    if (draft_kind != OR_DRAFT_POINT && draft == NULL) return -1;
    if (draft_kind == OR_DRAFT_LOGITS && draft_dtype != OR_F32 && draft_dtype != OR_BF16)
        return -1;
    outputs o = {accept_len, out_tokens, kv_commit, bonus, status};
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int b = 0; b < B; b++) {
        const int32_t *tok = draft_token + (size_t)b * N;
        const int32_t *par = parent + (size_t)b * N;
        const float *u = uniforms + (size_t)b * (N + 1);
        decision_margin[b] = INFINITY;
        cdf_margin[b] = INFINITY;
        cdf_alt[b] = -1;
        cdf_window[2 * b] = cdf_window[2 * b + 1] = -1;
        degenerate[b] = 0;
        if (T == 0.0) {
            greedy_one(logits, dtype, b, N, V, tok, par, o);
            continue;
        }
        int32_t st = check_request(par, tok, N, V);
        if (st == OR_OK)
            for (int i = 1; i <= N; i++)
                if (!(u[i] >= 0.0f && u[i] < 1.0f)) st = OR_BAD_UNIFORM;
        if (st != OR_OK) {
            write_failed(o, b, N, st);
            continue;
        }
        scratch s;
        s.p = (double *)malloc(sizeof(double) * (size_t)V);
        s.r = (double *)malloc(sizeof(double) * (size_t)V);
        s.q = (double *)malloc(sizeof(double) * (size_t)V);
        s.tmp = (double *)malloc((size_t)V + 8);
        int path[64], L = 0;
        int32_t res;
        if (draft_kind == OR_DRAFT_POINT)
            res = sample_point(logits, dtype, b, N, V, T, tok, par, u, s, path, &L,
                               &decision_margin[b], &cdf_margin[b], &cdf_alt[b],
                               &cdf_window[2 * b]);
        else
            res = sample_dense(logits, dtype, b, N, V, T, tok, par, draft, draft_kind,
                               draft_dtype, u, s, path, &L, &decision_margin[b],
                               &cdf_margin[b], &degenerate[b], &cdf_alt[b],
                               &cdf_window[2 * b]);
        if (res < 0)
            write_failed(o, b, N, -res);
        else
            write_path(o, b, N, tok, path, L, res);
        free(s.p);
        free(s.r);
        free(s.q);
        free(s.tmp);
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
