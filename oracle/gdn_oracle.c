/*
 * Token-by-token fp64 oracle for the gated delta rule (GDN scalar gate and
 * KDA per-key-channel gate).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do. It shares no code, header, table or constant with the CUDA
 * library.
 *
 * What it computes (the plain definition, one token at a time, no chunks):
 *
 *   Recurrence (the gated delta rule; for the
 *   per-key gate, decay first, as the state-summary page applies the decay
 *   to the state before the rank-one correction -- "state_summary.py",
 *   kda_split_state_summary_kernel loop body):
 *     a_t        = exp(g_t)  or 2^(g_t)     (per head, or per key channel)
 *     S'_t       = Diag(a_t) S_{t-1}
 *     e_t        = v_t - S'_t^T k_t
 *     S_t        = S'_t + beta_t k_t e_t^T
 *     o_t        = scale * S_t^T q_t
 *   so S_t = (I - beta_t k_t k_t^T) Diag(a_t) S_{t-1} + beta_t k_t v_t^T.
 *   The state is [K, V] (key-major, "state_v_first=False" in the Ascend C GDN
 *   adapter's forward call). The state restarts at h0 (or zero) at every
 *   document start.
 *
 *   Reverse mode: the exact adjoint of the steps above, token by token, with
 *   the state recomputed from checkpoints every 64 tokens.
 *
 *   Segment summary: S_ext = the recurrence from a zero state over one
 *   segment; M = the product of the per-token maps (I - b k k^T) Diag(a),
 *   i.e. the same recurrence run on the K columns of I with v = 0
 *   ("state_summary.py", kda_split_state_summary_kernel combined mode and
 *   kda_state_transition_kernel).
 *
 *   Merge: S_init_0 = h0 (or 0), S_init_{s+1} = M_s S_init_s + S_ext_s
 *   (apply_kda_state_summary on the coverage-diff page; SANA
 *   distributed_scan.py, _exclusive_prefix_compose).
 *
 * Layout of every token tensor: row-major [rows, H, D] where rows = B*T
 * (padded batch) or the packed token count (B == 1, cu != NULL).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t B, T, H, K, V;
    int32_t per_key;   /* 0: g is [rows, H]; 1: g is [rows, H, K] */
    int32_t use_exp2;  /* 0: a = exp(g); 1: a = 2^g */
    double scale;
    int64_t n_seq;     /* packed documents (cu != NULL), else ignored */
    const int64_t *cu; /* [n_seq + 1] document offsets, or NULL for padded batch */
    int32_t n_threads;
} orc_problem;

static int64_t n_units(const orc_problem *p) {
    return (p->cu ? p->n_seq : p->B) * p->H;
}

/* token range [*r0, *r1) in flattened rows, and the sequence index */
static void unit_range(const orc_problem *p, int64_t u, int64_t *seq, int64_t *h,
                       int64_t *r0, int64_t *r1) {
    *seq = u / p->H;
    *h = u % p->H;
    if (p->cu) {
        *r0 = p->cu[*seq];
        *r1 = p->cu[*seq + 1];
    } else {
        *r0 = *seq * p->T;
        *r1 = *r0 + p->T;
    }
}

static void decay_vector(const orc_problem *p, const double *g, int64_t row, int64_t h,
                         double *a) {
    for (int64_t d = 0; d < p->K; ++d) {
        double x = p->per_key ? g[(row * p->H + h) * p->K + d] : g[row * p->H + h];
        a[d] = p->use_exp2 ? exp2(x) : exp(x);
    }
}

/* One forward token step on state S [K, W]: S' = Diag(a) S, e = v - S'^T k,
 * S = S' + beta k e^T. v may be NULL (v = 0). If Sp is non-NULL it receives S'.
 */
static void token_step(int64_t K, int64_t W, const double *a, const double *k,
                       const double *v, double beta, double *S, double *e, double *Sp) {
    for (int64_t d = 0; d < K; ++d)
        for (int64_t c = 0; c < W; ++c) S[d * W + c] *= a[d];
    if (Sp) memcpy(Sp, S, sizeof(double) * K * W);
    for (int64_t c = 0; c < W; ++c) {
        double acc = 0.0;
        for (int64_t d = 0; d < K; ++d) acc += S[d * W + c] * k[d];
        e[c] = (v ? v[c] : 0.0) - acc;
    }
    for (int64_t d = 0; d < K; ++d)
        for (int64_t c = 0; c < W; ++c) S[d * W + c] += beta * k[d] * e[c];
}

/* ------------------------------------------------------------------ */
/* thread pool over independent units                                 */

typedef struct {
    const orc_problem *p;
    void (*fn)(const orc_problem *, int64_t, void *);
    void *arg;
    int64_t first, stride, count;
} orc_job;

static void *orc_worker(void *x) {
    orc_job *j = (orc_job *)x;
    for (int64_t u = j->first; u < j->count; u += j->stride) j->fn(j->p, u, j->arg);
    return NULL;
}

static void run_units(const orc_problem *p, int64_t count,
                      void (*fn)(const orc_problem *, int64_t, void *), void *arg) {
    int nt = p->n_threads > 0 ? p->n_threads : 1;
    if (nt > count) nt = (int)(count > 0 ? count : 1);
    if (nt <= 1) {
        for (int64_t u = 0; u < count; ++u) fn(p, u, arg);
        return;
    }
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    orc_job *jobs = (orc_job *)calloc((size_t)nt, sizeof(orc_job));
    for (int i = 0; i < nt; ++i) {
        jobs[i].p = p;
        jobs[i].fn = fn;
        jobs[i].arg = arg;
        jobs[i].first = i;
        jobs[i].stride = nt;
        jobs[i].count = count;
        pthread_create(&th[i], NULL, orc_worker, &jobs[i]);
    }
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    free(jobs);
}

/* ------------------------------------------------------------------ */
/* forward                                                            */

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0;
    double *o, *ht;
} fwd_args;

static void fwd_unit(const orc_problem *p, int64_t u, void *x) {
    fwd_args *A = (fwd_args *)x;
    const int64_t K = p->K, V = p->V, H = p->H;
    int64_t seq, h, r0, r1;
    unit_range(p, u, &seq, &h, &r0, &r1);
    double *S = (double *)calloc((size_t)(K * V), sizeof(double));
    double *a = (double *)malloc(sizeof(double) * K);
    double *e = (double *)malloc(sizeof(double) * V);
    if (A->h0) memcpy(S, A->h0 + (seq * H + h) * K * V, sizeof(double) * K * V);
    for (int64_t r = r0; r < r1; ++r) {
        decay_vector(p, A->g, r, h, a);
        const double *kr = A->k + (r * H + h) * K;
        const double *vr = A->v + (r * H + h) * V;
        const double *qr = A->q + (r * H + h) * K;
        token_step(K, V, a, kr, vr, A->beta[r * H + h], S, e, NULL);
        if (A->o) {
            double *orow = A->o + (r * H + h) * V;
            for (int64_t c = 0; c < V; ++c) {
                double acc = 0.0;
                for (int64_t d = 0; d < K; ++d) acc += S[d * V + c] * qr[d];
                orow[c] = p->scale * acc;
            }
        }
    }
    if (A->ht) memcpy(A->ht + (seq * H + h) * K * V, S, sizeof(double) * K * V);
    free(S);
    free(a);
    free(e);
}

int orc_forward(const orc_problem *p, const double *q, const double *k, const double *v,
                const double *g, const double *beta, const double *h0, double *o,
                double *ht) {
    fwd_args A = {q, k, v, g, beta, h0, o, ht};
    run_units(p, n_units(p), fwd_unit, &A);
    return 0;
}

/* ------------------------------------------------------------------ */
/* reverse mode                                                       */

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0, *dO, *dht;
    double *dq, *dk, *dv, *dg, *dbeta, *dh0;
} bwd_args;

#define ORC_CKPT 64

static void bwd_unit(const orc_problem *p, int64_t u, void *x) {
    bwd_args *A = (bwd_args *)x;
    const int64_t K = p->K, V = p->V, H = p->H, KV = p->K * p->V;
    int64_t seq, h, r0, r1;
    unit_range(p, u, &seq, &h, &r0, &r1);
    const int64_t L = r1 - r0;
    const int64_t nb = (L + ORC_CKPT - 1) / ORC_CKPT;
    double *ck = (double *)calloc((size_t)((nb > 0 ? nb : 1) * KV), sizeof(double));
    double *prev = (double *)malloc(sizeof(double) * ORC_CKPT * KV); /* S_{t-1} per token */
    double *S = (double *)calloc((size_t)KV, sizeof(double));
    double *Sp = (double *)malloc(sizeof(double) * KV);
    double *dS = (double *)calloc((size_t)KV, sizeof(double));
    double *a = (double *)malloc(sizeof(double) * K);
    double *e = (double *)malloc(sizeof(double) * V);
    double *de = (double *)malloc(sizeof(double) * V);
    const double ln2 = log(2.0);

    /* forward sweep, checkpointing the state before every block */
    if (A->h0) memcpy(S, A->h0 + (seq * H + h) * KV, sizeof(double) * KV);
    for (int64_t t = 0; t < L; ++t) {
        if (t % ORC_CKPT == 0) memcpy(ck + (t / ORC_CKPT) * KV, S, sizeof(double) * KV);
        int64_t r = r0 + t;
        decay_vector(p, A->g, r, h, a);
        token_step(K, V, a, A->k + (r * H + h) * K, A->v + (r * H + h) * V,
                   A->beta[r * H + h], S, e, NULL);
    }
    if (A->dht) memcpy(dS, A->dht + (seq * H + h) * KV, sizeof(double) * KV);

    for (int64_t b = nb - 1; b >= 0; --b) {
        int64_t t0 = b * ORC_CKPT, t1 = t0 + ORC_CKPT < L ? t0 + ORC_CKPT : L;
        memcpy(S, ck + b * KV, sizeof(double) * KV);
        for (int64_t t = t0; t < t1; ++t) {
            int64_t r = r0 + t;
            memcpy(prev + (t - t0) * KV, S, sizeof(double) * KV);
            decay_vector(p, A->g, r, h, a);
            token_step(K, V, a, A->k + (r * H + h) * K, A->v + (r * H + h) * V,
                       A->beta[r * H + h], S, e, NULL);
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            int64_t r = r0 + t;
            const double *kr = A->k + (r * H + h) * K;
            const double *qr = A->q + (r * H + h) * K;
            const double *vr = A->v + (r * H + h) * V;
            const double *dor = A->dO ? A->dO + (r * H + h) * V : NULL;
            const double bt = A->beta[r * H + h];
            /* recompute S'_t, e_t, S_t from S_{t-1} */
            memcpy(S, prev + (t - t0) * KV, sizeof(double) * KV);
            decay_vector(p, A->g, r, h, a);
            token_step(K, V, a, kr, vr, bt, S, e, Sp);
            /* o_t = scale S_t^T q_t */
            double *dqr = A->dq + (r * H + h) * K;
            for (int64_t d = 0; d < K; ++d) {
                double acc = 0.0;
                if (dor)
                    for (int64_t c = 0; c < V; ++c) acc += S[d * V + c] * dor[c];
                dqr[d] = p->scale * acc;
            }
            if (dor)
                for (int64_t d = 0; d < K; ++d)
                    for (int64_t c = 0; c < V; ++c) dS[d * V + c] += p->scale * qr[d] * dor[c];
            /* S_t = S'_t + beta k e^T */
            double dbeta = 0.0;
            double *dkr = A->dk + (r * H + h) * K;
            for (int64_t c = 0; c < V; ++c) {
                double acc = 0.0;
                for (int64_t d = 0; d < K; ++d) acc += dS[d * V + c] * kr[d];
                de[c] = bt * acc;
            }
            for (int64_t d = 0; d < K; ++d) {
                double acc = 0.0;
                for (int64_t c = 0; c < V; ++c) acc += dS[d * V + c] * e[c];
                dbeta += kr[d] * acc;
                dkr[d] = bt * acc;
            }
            A->dbeta[r * H + h] = dbeta;
            /* e = v - S'^T k */
            double *dvr = A->dv + (r * H + h) * V;
            for (int64_t c = 0; c < V; ++c) dvr[c] = de[c];
            for (int64_t d = 0; d < K; ++d) {
                double acc = 0.0;
                for (int64_t c = 0; c < V; ++c) acc += Sp[d * V + c] * de[c];
                dkr[d] -= acc;
            }
            for (int64_t d = 0; d < K; ++d)
                for (int64_t c = 0; c < V; ++c) dS[d * V + c] -= kr[d] * de[c]; /* dS' */
            /* S' = Diag(a) S_{t-1} */
            double gsum = 0.0;
            for (int64_t d = 0; d < K; ++d) {
                double acc = 0.0;
                for (int64_t c = 0; c < V; ++c) acc += dS[d * V + c] * Sp[d * V + c];
                if (p->use_exp2) acc *= ln2;
                if (p->per_key)
                    A->dg[(r * H + h) * K + d] = acc;
                else
                    gsum += acc;
            }
            if (!p->per_key) A->dg[r * H + h] = gsum;
            for (int64_t d = 0; d < K; ++d)
                for (int64_t c = 0; c < V; ++c) dS[d * V + c] *= a[d];
        }
    }
    if (A->dh0) memcpy(A->dh0 + (seq * H + h) * KV, dS, sizeof(double) * KV);
    free(ck);
    free(prev);
    free(S);
    free(Sp);
    free(dS);
    free(a);
    free(e);
    free(de);
}

int orc_backward(const orc_problem *p, const double *q, const double *k, const double *v,
                 const double *g, const double *beta, const double *h0, const double *dO,
                 const double *dht, double *dq, double *dk, double *dv, double *dg,
                 double *dbeta, double *dh0) {
    bwd_args A = {q, k, v, g, beta, h0, dO, dht, dq, dk, dv, dg, dbeta, dh0};
    run_units(p, n_units(p), bwd_unit, &A);
    return 0;
}

/* ------------------------------------------------------------------ */
/* segment summaries and merge (padded batch layout only)             */

typedef struct {
    const double *k, *v, *g, *beta;
    int64_t seg_len, nseg;
    double *S_ext, *M;
} sum_args;

static void sum_unit(const orc_problem *p, int64_t u, void *x) {
    sum_args *A = (sum_args *)x;
    const int64_t K = p->K, V = p->V, H = p->H;
    const int64_t b = u / (H * A->nseg), h = (u / A->nseg) % H, s = u % A->nseg;
    const int64_t t0 = s * A->seg_len;
    const int64_t t1 = t0 + A->seg_len < p->T ? t0 + A->seg_len : p->T;
    double *S = A->S_ext + ((b * H + h) * A->nseg + s) * K * V;
    double *M = A->M + ((b * H + h) * A->nseg + s) * K * K;
    double *a = (double *)malloc(sizeof(double) * K);
    double *e = (double *)malloc(sizeof(double) * (V > K ? V : K));
    memset(S, 0, sizeof(double) * K * V);
    memset(M, 0, sizeof(double) * K * K);
    for (int64_t d = 0; d < K; ++d) M[d * K + d] = 1.0;
    for (int64_t t = t0; t < t1; ++t) {
        int64_t r = b * p->T + t;
        decay_vector(p, A->g, r, h, a);
        const double *kr = A->k + (r * H + h) * K;
        const double bt = A->beta[r * H + h];
        token_step(K, V, a, kr, A->v + (r * H + h) * V, bt, S, e, NULL);
        token_step(K, K, a, kr, NULL, bt, M, e, NULL);
    }
    free(a);
    free(e);
}

int orc_segment_summary(const orc_problem *p, const double *k, const double *v,
                        const double *g, const double *beta, int64_t seg_len,
                        double *S_ext, double *M) {
    if (p->cu || seg_len <= 0) return 1;
    sum_args A = {k, v, g, beta, seg_len, (p->T + seg_len - 1) / seg_len, S_ext, M};
    run_units(p, p->B * p->H * A.nseg, sum_unit, &A);
    return 0;
}

/* S_init [B,H,nseg,K,V]: entry state of each segment; ht [B,H,K,V] (nullable) */
int orc_segment_merge(const orc_problem *p, const double *S_ext, const double *M,
                      int64_t nseg, const double *h0, double *S_init, double *ht) {
    const int64_t K = p->K, V = p->V, H = p->H;
    double *cur = (double *)malloc(sizeof(double) * K * V);
    double *nxt = (double *)malloc(sizeof(double) * K * V);
    for (int64_t bh = 0; bh < p->B * H; ++bh) {
        if (h0)
            memcpy(cur, h0 + bh * K * V, sizeof(double) * K * V);
        else
            memset(cur, 0, sizeof(double) * K * V);
        for (int64_t s = 0; s < nseg; ++s) {
            memcpy(S_init + (bh * nseg + s) * K * V, cur, sizeof(double) * K * V);
            const double *Ms = M + (bh * nseg + s) * K * K;
            const double *Es = S_ext + (bh * nseg + s) * K * V;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t c = 0; c < V; ++c) {
                    double acc = Es[i * V + c];
                    for (int64_t j = 0; j < K; ++j) acc += Ms[i * K + j] * cur[j * V + c];
                    nxt[i * V + c] = acc;
                }
            memcpy(cur, nxt, sizeof(double) * K * V);
        }
        if (ht) memcpy(ht + bh * K * V, cur, sizeof(double) * K * V);
    }
    free(cur);
    free(nxt);
    return 0;
}
