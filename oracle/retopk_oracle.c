/*
 * retopk_oracle.c -- plain, slow fp64 CPU oracle for ReTopK and Exact Top-K
 * decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this code:
 * only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no source with the CUDA library.
 *
 * Method: "Recall Before You Rank: Similarity-Guided Top-K Reuse for Efficient
 * Long-Context Attention" (ReTopK).  Each function names the equation it
 * follows; sections are those of that paper:
 *   §Motivation               Eq. (1)  Exact Top-K support;
 *                             Eqs. (2)-(3) support overlap and coverage
 *                                        (diagnostics of support reuse)
 *   §Problem Setup            Eq. (4)  full-history scores
 *   §Recall-Before-Rerank     Eqs. (5)-(12)  cache, recall, candidates,
 *                                        rerank, reranked support, sparse
 *                                        softmax-value aggregation
 *   §Reliable Reuse           Eq. (13) path rule; cache insertion after either
 *                                        path
 * and the softmax merge of two disjoint partial attentions from the
 * RetrievalAttention notes (§3, Appendix B Eqs. (3)-(5)).
 *
 * Everything is computed in double precision from the exact values of the bf16
 * inputs.  Indices are 0-based: the paper's key i (1-based) is key i-1 here,
 * and its recent window {max(1, L-W+1), ..., L} is {max(0, L-W), ..., L-1}.
 *
 * Readings taken where the paper is silent (each one is listed with its
 * reason in the project's design notes):
 *   - L counts the current token, whose key/value is appended before the step.
 *   - Top-K / Top-R ties: a lower key index (older cache entry) ranks first.
 *   - Fewer than K candidates (or keys): the support is all of them.
 *   - Path rule: refresh when T_r > 0 and t_dec is a multiple of T_r, where
 *     the first decode step has t_dec = 1; otherwise fall back when
 *     rho_max < tau (strict); otherwise reuse.  An empty cache, or a zero
 *     query norm, gives rho = -inf and so falls back.
 *   - The cache stores the raw bf16 query (normalisation is applied when the
 *     cosine is taken, Eq. (6) written as D(a,b)/sqrt(D(a,a) D(b,b))) and the
 *     support as an ascending index list with its length.
 *   - Cache initialisation: prompt position p in [L0-C, L0-1] stores its query
 *     and the exact Top-K of that query over the causal prefix 0..p.
 *   - Softmax is max-shifted (mathematically identical to Eq. (12)).
 *
 * Parity is pinned by the tests in tests/test_oracle_pins.py (closed forms,
 * brute force, library routines and the paper's stated invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* exact widening of a bf16 bit pattern */
static double bf(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double dot_bf(const uint16_t *a, const uint16_t *b, int d)
{
    double s = 0.0;
    for (int j = 0; j < d; ++j)
        s += bf(a[j]) * bf(b[j]);
    return s;
}

/* ------------------------------------------------------------------------ */
/* Eq. (4) / Eq. (10): e_i = q . k_i / sqrt(d) for the listed keys.          */
/* keys are rows of `k` (row stride `ld` elements); idx == NULL means 0..n-1. */
void oracle_scores(const uint16_t *q, const uint16_t *k, int64_t ld,
                   const int32_t *idx, int n, int d, double *out)
{
    double inv = 1.0 / sqrt((double)d);
    for (int j = 0; j < n; ++j) {
        int64_t i = idx ? idx[j] : j;
        out[j] = dot_bf(q, k + i * ld, d) * inv;
    }
}

/* ------------------------------------------------------------------------ */
/* Eqs. (1), (11): Top-K.  Orders (score, index) pairs by score descending,  */
/* then index ascending, and keeps the first min(K, n).                      */
typedef struct { double s; int32_t i; } pair_t;

static int cmp_pair(const void *a, const void *b)
{
    const pair_t *x = (const pair_t *)a, *y = (const pair_t *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Writes the selected indices in rank order (best first); returns the count. */
int oracle_topk(const double *score, const int32_t *idx, int n, int K, int32_t *out)
{
    pair_t *p = (pair_t *)malloc(sizeof(pair_t) * (size_t)(n > 0 ? n : 1));
    for (int j = 0; j < n; ++j) {
        p[j].s = score[j];
        p[j].i = idx ? idx[j] : j;
    }
    qsort(p, (size_t)n, sizeof(pair_t), cmp_pair);
    int m = n < K ? n : K;
    for (int j = 0; j < m; ++j)
        out[j] = p[j].i;
    free(p);
    return m;
}

/* ------------------------------------------------------------------------ */
/* Eq. (12): softmax over the support's scores, then the weighted sum of the */
/* value rows.  `score[j]` belongs to key `idx[j]`.                          */
void oracle_sparse_attention(const double *score, const int32_t *idx, int n,
                             const uint16_t *v, int64_t ld, int d, double *out)
{
    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    if (n <= 0)
        return;
    double m = score[0];
    for (int j = 1; j < n; ++j)
        if (score[j] > m) m = score[j];
    double Z = 0.0;
    for (int j = 0; j < n; ++j)
        Z += exp(score[j] - m);
    for (int j = 0; j < n; ++j) {
        double w = exp(score[j] - m) / Z;
        const uint16_t *row = v + (int64_t)idx[j] * ld;
        for (int c = 0; c < d; ++c)
            out[c] += w * bf(row[c]);
    }
}

/* Attention on a given support: scores by Eq. (10), weights by Eq. (12).    */
void oracle_attention_on_support(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 int64_t ld, const int32_t *sup, int n, int d, double *out)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    oracle_scores(q, k, ld, sup, n, d, s);
    oracle_sparse_attention(s, sup, n, v, ld, d, out);
    free(s);
}

/* Dense softmax attention over keys 0..L-1 (used only to pin the K >= L case). */
void oracle_dense_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            int64_t ld, int L, int d, double *out)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    int32_t *all = (int32_t *)malloc(sizeof(int32_t) * (size_t)(L > 0 ? L : 1));
    oracle_scores(q, k, ld, NULL, L, d, s);
    for (int i = 0; i < L; ++i)
        all[i] = i;
    oracle_sparse_attention(s, all, L, v, ld, d, out);
    free(all);
    free(s);
}

/* ------------------------------------------------------------------------ */
/* Softmax merge of two disjoint partial attentions (RetrievalAttention      */
/* notes, §3 / Appendix B Eqs. (3)-(5)): part S carries its max m_S, its     */
/* shifted normaliser Z_S = sum exp(z - m_S) and its normalised output o_S;  */
/* with m = max(m_1, m_2), gamma_S = exp(m_S - m) Z_S / sum_S' exp(m_S' - m) Z_S'. */
void oracle_softmax_merge(double m1, double Z1, const double *o1,
                          double m2, double Z2, const double *o2,
                          int d, double *m_out, double *Z_out, double *o_out)
{
    double m = m1 > m2 ? m1 : m2;
    double a1 = exp(m1 - m) * Z1, a2 = exp(m2 - m) * Z2;
    double g1 = a1 / (a1 + a2), g2 = a2 / (a1 + a2);
    for (int c = 0; c < d; ++c)
        o_out[c] = g1 * o1[c] + g2 * o2[c];
    *m_out = m;
    *Z_out = a1 + a2;
}

/* ------------------------------------------------------------------------ */
/* Eqs. (6)-(7): cosine recall against the n cached queries (oldest first).  */
/* rho[c] = D(q, q_c) / sqrt(D(q,q) D(q_c,q_c)); a zero norm gives -inf.     */
/* topR receives min(R, n) logical positions ordered by (rho desc, age asc); */
/* the return value is rho_max (-inf when n == 0).                          */
double oracle_recall(const uint16_t *q, const uint16_t *const *cached, int n, int d,
                     int R, double *rho, int32_t *topR)
{
    double nq = dot_bf(q, q, d);
    pair_t *p = (pair_t *)malloc(sizeof(pair_t) * (size_t)(n > 0 ? n : 1));
    for (int c = 0; c < n; ++c) {
        double nc = dot_bf(cached[c], cached[c], d);
        double r = (nq > 0.0 && nc > 0.0) ? dot_bf(q, cached[c], d) / sqrt(nq * nc) : -INFINITY;
        rho[c] = r;
        p[c].s = r;
        p[c].i = c;
    }
    qsort(p, (size_t)n, sizeof(pair_t), cmp_pair);
    int m = n < R ? n : R;
    for (int r = 0; r < m; ++r)
        topR[r] = p[r].i;
    for (int r = m; r < R; ++r)
        topR[r] = -1;
    double rmax = n > 0 ? p[0].s : -INFINITY;
    free(p);
    return rmax;
}

/* ------------------------------------------------------------------------ */
/* Eqs. (8)-(9): A_t = Unique(union of the retrieved supports and the recent */
/* window {max(0, L-W) .. L-1}), written in ascending order.  Returns M_t.   */
int oracle_candidates(const int32_t *const *sup, const int32_t *len, int nsup,
                      int L, int W, int32_t *out)
{
    int total = 0;
    for (int r = 0; r < nsup; ++r)
        total += len[r];
    int lo = L - W > 0 ? L - W : 0;
    total += L - lo;
    int32_t *all = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total > 0 ? total : 1));
    int n = 0;
    for (int i = lo; i < L; ++i)
        all[n++] = i;
    for (int r = 0; r < nsup; ++r)
        for (int j = 0; j < len[r]; ++j)
            all[n++] = sup[r][j];
    qsort(all, (size_t)n, sizeof(int32_t), cmp_i32);
    int M = 0;
    for (int j = 0; j < n; ++j)
        if (M == 0 || all[j] != out[M - 1])
            out[M++] = all[j];
    free(all);
    return M;
}

/* ------------------------------------------------------------------------ */
/* Exact Top-K attention for one query over keys 0..L-1 (Eqs. (1), (4), (12)). */
/* Writes the support in ascending index order; returns its length.          */
/* kth_score receives the score of the last selected key (or -inf).          */
int oracle_exact_one(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t ld,
                     int L, int d, int K, int32_t *sup, double *kth_score, double *out)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    oracle_scores(q, k, ld, NULL, L, d, s);
    int n = oracle_topk(s, NULL, L, K, sup);
    if (kth_score)
        *kth_score = n > 0 ? s[sup[n - 1]] : -INFINITY;
    qsort(sup, (size_t)n, sizeof(int32_t), cmp_i32);
    if (out) {
        double *ss = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        for (int j = 0; j < n; ++j)
            ss[j] = s[sup[j]];
        oracle_sparse_attention(ss, sup, n, v, ld, d, out);
        free(ss);
    }
    free(s);
    return n;
}

/* Batched Exact Top-K step (the stateless comparison path).                 */
/* q [B,Hq,d]; k,v [B,Hkv,ld_len,d]; L[B]; sup [B,Hq,K] (-1 padded);         */
/* sup_len [B,Hq]; kth [B,Hq]; out [B,Hq,d].                                 */
void oracle_exact_step(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *L, int B, int Hq, int Hkv, int d, int64_t max_len,
                       int K, int32_t *sup, int32_t *sup_len, double *kth, double *out)
{
    int G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hq; ++bh) {
        int b = bh / Hq, h = bh % Hq, hk = h / G;
        const uint16_t *kb = k + ((int64_t)b * Hkv + hk) * max_len * d;
        const uint16_t *vb = v + ((int64_t)b * Hkv + hk) * max_len * d;
        int32_t *s = sup + (int64_t)bh * K;
        for (int j = 0; j < K; ++j)
            s[j] = -1;
        sup_len[bh] = oracle_exact_one(q + (int64_t)bh * d, kb, vb, d, L[b], d, K, s,
                                       kth + bh, out + (int64_t)bh * d);
    }
}

/* ------------------------------------------------------------------------ */
/* Query-support cache of one sequence (Eq. (5)), FIFO of capacity C per     */
/* query head:  fq [Hq,C,d] raw bf16 queries, fsup [Hq,C,K] ascending       */
/* supports, flen [Hq,C] support lengths, seq[0] = next slot to write,      */
/* seq[1] = number of live entries, seq[2] = decode steps taken so far.      */
/* Live entry c (0 = oldest) sits in slot (seq[0] - seq[1] + c) mod C.       */

/* Cache initialisation from the final C prompt queries (one sequence).      */
/* qp [Hq,C,d] holds the queries of prompt positions L0-C .. L0-1.           */
int oracle_init_cache(const uint16_t *qp, const uint16_t *k, int64_t max_len, int L0,
                      int Hq, int Hkv, int d, int K, int C,
                      uint16_t *fq, int32_t *fsup, int32_t *flen, int32_t *seq)
{
    if (L0 < C || C < 1)
        return -1;
    int G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int hc = 0; hc < Hq * C; ++hc) {
        int h = hc / C, c = hc % C;
        int p = L0 - C + c;
        const uint16_t *qq = qp + ((int64_t)h * C + c) * d;
        const uint16_t *kb = k + (int64_t)(h / G) * max_len * d;
        int32_t *s = fsup + ((int64_t)h * C + c) * K;
        for (int j = 0; j < K; ++j)
            s[j] = -1;
        flen[h * C + c] = oracle_exact_one(qq, kb, NULL, d, p + 1, d, K, s, NULL, NULL);
        memcpy(fq + ((int64_t)h * C + c) * d, qq, sizeof(uint16_t) * (size_t)d);
    }
    seq[0] = 0;          /* C insertions into an empty ring of size C wrap to 0 */
    seq[1] = C;
    seq[2] = 0;
    return 0;
}

/* One ReTopK decode step for one sequence (all query heads).                 */
/* Inputs: q [Hq,d]; k, v [Hkv,max_len,d]; L keys (current one included).     */
/* Cache state fq/fsup/flen/seq is read before and updated after the step.    */
/* Outputs per head h:                                                        */
/*   path[h]    0 reuse, 1 exact by similarity fallback, 2 exact by refresh   */
/*   rho[h*C+c] cosine to live entry c (oldest first); unused entries NaN     */
/*   rho_max[h], topR[h*R+r] (logical entry positions, -1 padded)             */
/*   cand[h*cap+j], M[h]: A_t ascending on reuse steps (M = L, cand unset on  */
/*                        exact steps)                                        */
/*   sup[h*K+j], sup_len[h]: the selected support, ascending (-1 padded)      */
/*   kth[h]     score of the K-th ranked key of the support                   */
/*   out[h*d+c] Eq. (12) output                                               */
/* The ablation the paper's Table 3 calls "recent-R retrieval": the R most
 * recent live entries (newest first) instead of the R most similar, with
 * rho_max taken over them.  rho: every entry's cosine, as for Eq. (6). */
double oracle_recall_recent(const uint16_t *q, const uint16_t *const *cached, int n, int d,
                            int R, double *rho, int32_t *topR)
{
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    oracle_recall(q, cached, n, d, R, rho, tmp);   /* the cosines */
    free(tmp);
    int m = n < R ? n : R;
    double rmax = -INFINITY;
    for (int r = 0; r < m; ++r) {
        topR[r] = n - 1 - r;
        if (rho[n - 1 - r] > rmax)
            rmax = rho[n - 1 - r];
    }
    for (int r = m; r < R; ++r)
        topR[r] = -1;
    return rmax;
}

void oracle_decode_step(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        int64_t max_len, int L, int Hq, int Hkv, int d,
                        int K, int C, int W, int R, int T_r, double tau, int recent,
                        uint16_t *fq, int32_t *fsup, int32_t *flen, int32_t *seq,
                        int32_t *path, double *rho, double *rho_max, int32_t *topR,
                        int32_t *cand, int cap, int32_t *M,
                        int32_t *sup, int32_t *sup_len, double *kth, double *out)
{
    int G = Hq / Hkv;
    int head = seq[0], count = seq[1];
    int t_dec = seq[2] + 1;                          /* this step's decode offset */
    int refresh = (T_r > 0) && (t_dec % T_r == 0);  /* Eq. (13), first case      */
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < Hq; ++h) {
        const uint16_t *qh = q + (int64_t)h * d;
        const uint16_t *kb = k + (int64_t)(h / G) * max_len * d;
        const uint16_t *vb = v + (int64_t)(h / G) * max_len * d;
        int32_t *s = sup + (int64_t)h * K;
        for (int j = 0; j < K; ++j)
            s[j] = -1;
        /* Eqs. (6)-(7): recall against the cache as it stands (before insertion) */
        const uint16_t **cq = (const uint16_t **)malloc(sizeof(void *) * (size_t)(count > 0 ? count : 1));
        int *slot = (int *)malloc(sizeof(int) * (size_t)(count > 0 ? count : 1));
        for (int c = 0; c < count; ++c) {
            slot[c] = ((head - count + c) % C + C) % C;
            cq[c] = fq + ((int64_t)h * C + slot[c]) * d;
        }
        for (int c = 0; c < C; ++c)
            rho[(int64_t)h * C + c] = NAN;
        rho_max[h] = (recent ? oracle_recall_recent : oracle_recall)(qh, cq, count, d, R, rho + (int64_t)h * C,
                                                                  topR + (int64_t)h * R);
        /* Eq. (13) */
        int p = refresh ? 2 : (rho_max[h] < tau || isnan(rho_max[h])) ? 1 : 0;
        path[h] = p;
        if (p == 0) {
            /* Eqs. (8)-(9): candidate set from the retrieved supports and the window */
            const int32_t *sp[256];
            int32_t ln[256];
            int nsup = 0;
            for (int r = 0; r < R && r < count; ++r) {
                int sl = slot[topR[(int64_t)h * R + r]];
                sp[nsup] = fsup + ((int64_t)h * C + sl) * K;
                ln[nsup] = flen[h * C + sl];
                ++nsup;
            }
            int32_t *A = cand + (int64_t)h * cap;
            int m = oracle_candidates(sp, ln, nsup, L, W, A);
            M[h] = m;
            /* Eq. (10): exact scores of the candidates only; Eq. (11): Top-K */
            double *e = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
            oracle_scores(qh, kb, d, A, m, d, e);
            int n = oracle_topk(e, A, m, K, s);
            /* score of the K-th ranked key */
            double kk = -INFINITY;
            if (n > 0) {
                int32_t last = s[n - 1];
                for (int j = 0; j < m; ++j)
                    if (A[j] == last) { kk = e[j]; break; }
            }
            kth[h] = kk;
            qsort(s, (size_t)n, sizeof(int32_t), cmp_i32);
            sup_len[h] = n;
            /* Eq. (12) over the reranked support */
            double *es = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
            oracle_scores(qh, kb, d, s, n, d, es);
            oracle_sparse_attention(es, s, n, vb, d, d, out + (int64_t)h * d);
            free(es);
            free(e);
        } else {
            /* Exact Top-K over the full history (Eqs. (1), (4), (12)) */
            M[h] = L;
            sup_len[h] = oracle_exact_one(qh, kb, vb, d, L, d, K, s, kth + h, out + (int64_t)h * d);
        }
        free(slot);
        free(cq);
    }
    /* cache update after either path with (q_t, S_t) (§Reliable Reuse) */
    for (int h = 0; h < Hq; ++h) {
        memcpy(fq + ((int64_t)h * C + head) * d, q + (int64_t)h * d, sizeof(uint16_t) * (size_t)d);
        int32_t *dst = fsup + ((int64_t)h * C + head) * K;
        for (int j = 0; j < K; ++j)
            dst[j] = sup[(int64_t)h * K + j];
        flen[h * C + head] = sup_len[h];
    }
    seq[0] = (head + 1) % C;
    seq[1] = count + 1 < C ? count + 1 : C;
    seq[2] = t_dec;
}

/* Attention-support fidelity of a reuse support against the exact one
 * (ReTopK paper, §Experiments "Attention-support fidelity" with Figs. 5-6,
 * and §Motivation Eqs. (2)-(3) for the overlap of two supports).  S (nS keys)
 * is the Exact Top-K support of q, Sh (nh keys) the support being judged;
 * both ascending.  Scores are recomputed from q and the K rows; p and ph are
 * the softmax distributions over S and Sh.  out[0] = |Sh n S| / nS (support
 * recall, Eq. (2)'s overlap with nS = K), out[1] = sum of p over Sh n S (the
 * Exact Top-K attention mass the support retains), out[2] = cosine of the two
 * head outputs oh and o (d values each), out[3] = cosine of the two
 * attention distributions (sum over Sh n S of p ph / (|p| |ph|)). */
void oracle_fidelity(const uint16_t *q, const uint16_t *k, int64_t ld, int d,
                     const int32_t *S, int nS, const int32_t *Sh, int nh,
                     const double *o, const double *oh, double *out)
{
    double *eS = (double *)malloc(sizeof(double) * (nS > 0 ? nS : 1));
    double *eh = (double *)malloc(sizeof(double) * (nh > 0 ? nh : 1));
    oracle_scores(q, k, ld, S, nS, d, eS);
    oracle_scores(q, k, ld, Sh, nh, d, eh);
    double mS = -INFINITY, mh = -INFINITY, ZS = 0.0, Zh = 0.0, p2 = 0.0, ph2 = 0.0;
    for (int i = 0; i < nS; ++i)
        mS = fmax(mS, eS[i]);
    for (int i = 0; i < nh; ++i)
        mh = fmax(mh, eh[i]);
    for (int i = 0; i < nS; ++i)
        ZS += exp(eS[i] - mS);
    for (int i = 0; i < nh; ++i)
        Zh += exp(eh[i] - mh);
    for (int i = 0; i < nS; ++i)
        p2 += (exp(eS[i] - mS) / ZS) * (exp(eS[i] - mS) / ZS);
    for (int i = 0; i < nh; ++i)
        ph2 += (exp(eh[i] - mh) / Zh) * (exp(eh[i] - mh) / Zh);
    int common = 0;
    double mass = 0.0, cross = 0.0;
    for (int a = 0, b = 0; a < nS && b < nh;) {   /* both ascending: merge */
        if (S[a] < Sh[b]) {
            ++a;
        } else if (Sh[b] < S[a]) {
            ++b;
        } else {
            const double p = exp(eS[a] - mS) / ZS, ph = exp(eh[b] - mh) / Zh;
            ++common;
            mass += p;
            cross += p * ph;
            ++a;
            ++b;
        }
    }
    double oo = 0.0, hh = 0.0, oh2 = 0.0;
    for (int c = 0; c < d; ++c) {
        oo += o[c] * o[c];
        hh += oh[c] * oh[c];
        oh2 += o[c] * oh[c];
    }
    out[0] = nS > 0 ? (double)common / nS : 1.0;
    out[1] = mass;
    out[2] = (oo > 0.0 && hh > 0.0) ? oh2 / (sqrt(oo) * sqrt(hh)) : 0.0;
    out[3] = (p2 > 0.0 && ph2 > 0.0) ? cross / (sqrt(p2) * sqrt(ph2)) : 0.0;
    free(eS);
    free(eh);
}

/* §Motivation Eq. (2): the normalised overlap of two Exact Top-K supports,
 * |S_t n S_j| / K (both ascending; the denominator is K as printed, also when
 * a support is shorter than K because fewer keys exist). */
double oracle_overlap(const int32_t *St, int nt, const int32_t *Sj, int nj, int K)
{
    int common = 0;
    for (int a = 0, b = 0; a < nt && b < nj;) {
        if (St[a] < Sj[b])
            ++a;
        else if (Sj[b] < St[a])
            ++b;
        else {
            ++common;
            ++a;
            ++b;
        }
    }
    return (double)common / K;
}

/* §Motivation Eq. (3): Coverage_t(R) = |S_t n U_t(R)| / K, where U_t(R) is the
 * union of the supports of the R preceding queries most similar to q (cosine,
 * Eq. (6); ties to the older query, as for Eq. (7)).  prev_q / prev_S /
 * prev_n: the n_prev preceding queries, oldest first, with their ascending
 * supports.  chosen[0..R) receives the selected positions (-1 padded).
 * Returns the coverage. */
double oracle_coverage(const uint16_t *q, const uint16_t *const *prev_q, const int32_t *const *prev_S,
                       const int32_t *prev_n, int n_prev, int d, int R, const int32_t *St, int nt, int K,
                       int32_t *chosen)
{
    double *rho = (double *)malloc(sizeof(double) * (size_t)(n_prev > 0 ? n_prev : 1));
    oracle_recall(q, prev_q, n_prev, d, R, rho, chosen);
    const int m = n_prev < R ? n_prev : R;
    const int32_t *sp[256];
    int32_t ln[256];
    int total = 0;
    for (int r = 0; r < m && r < 256; ++r) {
        sp[r] = prev_S[chosen[r]];
        ln[r] = prev_n[chosen[r]];
        total += ln[r];
    }
    int32_t *U = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total > 0 ? total : 1));
    const int nu = oracle_candidates(sp, ln, m < 256 ? m : 256, 0, 0, U);   /* union only: no window */
    const double cov = oracle_overlap(St, nt, U, nu, K);
    free(U);
    free(rho);
    return cov;
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
