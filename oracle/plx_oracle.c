/*
 * Parallax attention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of the layer, written to be checked by eye
 * against its definition.  Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library; the CUDA library never
 * does, and the two share no code.
 *
 * Definition (per batch b and head h, causal: key index i <= query index t).
 * Source: "Parallax: Parameterized Local Linear Attention for Language
 * Modeling" (gist.science technical summary, "Core mechanism": the output is
 * the softmax-attention output plus a correction made of the KV covariance
 * applied to a learned probe; the boundary-amplification factor eta is set to
 * zero).  The probe here is rho_t = -u_t with u_t = P_h (q_t - mu_k,t), the
 * per-head learned d x d projector standing in for the inverse key covariance
 * that exact Local Linear Attention would solve for ("Problem statement").
 *
 *   s_ti  = c q_t . k_i,  c = 1/sqrt(d)
 *   L_t   = log sum_{i<=t} exp(s_ti)          (natural log, c included)
 *   p_ti  = exp(s_ti - L_t)
 *   mu_v  = sum_i p_ti v_i,   mu_k = sum_i p_ti k_i
 *   u_t   = P_h (q_t - mu_k)                  (P_h row-major: u[a] = sum_b P[a][b] delta[b])
 *   g_ti  = k_i . u_t,        gbar_t = sum_i p_ti g_ti
 *   o_t   = mu_v + sum_i p_ti g_ti v_i - gbar_t mu_v
 *
 * The last line is o^SA + Sigma_KV u with Sigma_KV = sum_i p_i (v_i - mu_v)(k_i - mu_k)^T,
 * the softmax-weighted cross-covariance (reading: the pages never spell out
 * Sigma_KV; centring both factors at the softmax means is what makes a zero
 * projector give softmax attention exactly, as the write-ups state).
 *
 * Backward: the chain rule of the lines above, written per query t
 * (e_i = do_t . v_i):
 *   ebar = sum p_i e_i;  a_i = p_i (1 + g_i - gbar);  dv_i += a_i do_t
 *   dg_i = p_i (e_i - ebar);  du = sum dg_i k_i;  dk_i += dg_i u
 *   dP_h += du delta^T;  ddelta = P_h^T du;  dq_t += ddelta;  dmu_k = -ddelta;
 *   dk_i += p_i dmu_k
 *   D = do . o - gbar ebar + mu_k . dmu_k
 *   ds_i = p_i (e_i (1 + g_i - gbar) - g_i ebar + k_i . dmu_k - D)
 *   dq_t += c sum ds_i k_i;  dk_i += c ds_i q_t
 *
 * Pins (tests/test_oracle_pins.py): P = 0 against a library softmax
 * attention; per-query P = (Sigma_kk + lambda I)^-1 against an independent
 * weighted-least-squares local-linear fit (exact LLA); constant values; the
 * probe-orientation subspace invariant; linearity in P; central finite
 * differences for every gradient.
 *
 * Layouts: q, k, v, dout, out, mu_k, dq, dk, dv are contiguous [B][H][T][d];
 * lse is [B][H][T]; P and dP are [H][d][d] (or [B][H][T][d][d] when
 * p_per_query != 0, a test hook for the exact-LLA check).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *P, *dout;
    int B, H, T, d, p_per_query;
} plx_in_t;

static const double *head_ptr(const double *x, const plx_in_t *in, int b, int h) {
    return x + ((size_t)b * in->H + h) * (size_t)in->T * in->d;
}

static const double *proj_ptr(const plx_in_t *in, int b, int h, int t) {
    size_t dd = (size_t)in->d * in->d;
    if (in->p_per_query)
        return in->P + (((size_t)b * in->H + h) * in->T + t) * dd;
    return in->P + (size_t)h * dd;
}

/* Per-query scratch: T scores/weights/g/e, plus d-vectors. */
typedef struct {
    double *s, *p, *g, *e, *mu_v, *mu_k, *delta, *u, *o;
    double *du, *ddelta, *dmu_k;
} scratch_t;

static int scratch_alloc(scratch_t *w, int T, int d) {
    memset(w, 0, sizeof(*w));
    w->s = malloc(sizeof(double) * (size_t)T);
    w->p = malloc(sizeof(double) * (size_t)T);
    w->g = malloc(sizeof(double) * (size_t)T);
    w->e = malloc(sizeof(double) * (size_t)T);
    w->mu_v = malloc(sizeof(double) * (size_t)d * 9);
    if (!w->s || !w->p || !w->g || !w->e || !w->mu_v) return -1;
    w->mu_k = w->mu_v + d;
    w->delta = w->mu_v + 2 * d;
    w->u = w->mu_v + 3 * d;
    w->o = w->mu_v + 4 * d;
    w->du = w->mu_v + 5 * d;
    w->ddelta = w->mu_v + 6 * d;
    w->dmu_k = w->mu_v + 7 * d;
    return 0;
}

static void scratch_free(scratch_t *w) {
    free(w->s); free(w->p); free(w->g); free(w->e); free(w->mu_v);
}

/* Forward for one query t of head (b,h); fills w->p, w->g, mu_v, mu_k, delta,
 * u, o and returns L_t.  Every sum is a plain left-to-right fp64 loop. */
static double forward_query(const plx_in_t *in, int b, int h, int t, scratch_t *w,
                            double *gbar_out) {
    const int d = in->d;
    const double c = 1.0 / sqrt((double)d);
    const double *Q = head_ptr(in->q, in, b, h);
    const double *K = head_ptr(in->k, in, b, h);
    const double *V = head_ptr(in->v, in, b, h);
    const double *qt = Q + (size_t)t * d;
    const double *P = proj_ptr(in, b, h, t);

    /* scores and softmax with max subtraction */
    double m = -INFINITY;
    for (int i = 0; i <= t; i++) {
        double acc = 0.0;
        for (int j = 0; j < d; j++) acc += qt[j] * K[(size_t)i * d + j];
        w->s[i] = c * acc;
        if (w->s[i] > m) m = w->s[i];
    }
    double Z = 0.0;
    for (int i = 0; i <= t; i++) Z += exp(w->s[i] - m);
    const double L = m + log(Z);
    for (int i = 0; i <= t; i++) w->p[i] = exp(w->s[i] - L);

    /* softmax means of values and keys */
    for (int j = 0; j < d; j++) { w->mu_v[j] = 0.0; w->mu_k[j] = 0.0; }
    for (int i = 0; i <= t; i++) {
        for (int j = 0; j < d; j++) {
            w->mu_v[j] += w->p[i] * V[(size_t)i * d + j];
            w->mu_k[j] += w->p[i] * K[(size_t)i * d + j];
        }
    }
    /* probe u = P (q - mu_k) */
    for (int j = 0; j < d; j++) w->delta[j] = qt[j] - w->mu_k[j];
    for (int a = 0; a < d; a++) {
        double acc = 0.0;
        for (int bb = 0; bb < d; bb++) acc += P[(size_t)a * d + bb] * w->delta[bb];
        w->u[a] = acc;
    }
    /* g_i = k_i . u and its softmax mean */
    double gbar = 0.0;
    for (int i = 0; i <= t; i++) {
        double acc = 0.0;
        for (int j = 0; j < d; j++) acc += K[(size_t)i * d + j] * w->u[j];
        w->g[i] = acc;
        gbar += w->p[i] * acc;
    }
    /* o = mu_v + sum p g v - gbar mu_v */
    for (int j = 0; j < d; j++) w->o[j] = 0.0;
    for (int i = 0; i <= t; i++) {
        const double pg = w->p[i] * w->g[i];
        for (int j = 0; j < d; j++) w->o[j] += pg * V[(size_t)i * d + j];
    }
    for (int j = 0; j < d; j++) w->o[j] = w->mu_v[j] + w->o[j] - gbar * w->mu_v[j];
    *gbar_out = gbar;
    return L;
}

/* ------------------------------------------------------------------ threads */

typedef struct {
    const plx_in_t *in;
    int njobs;
    int next;
    pthread_mutex_t mu;
    void (*run)(void *ctx, int job, scratch_t *w, double *dp);
    void *ctx;
    int failed;
    double *dp_partial; /* per job d*d (backward only) */
} pool_t;

static void *worker(void *arg) {
    pool_t *pool = (pool_t *)arg;
    scratch_t w;
    if (scratch_alloc(&w, pool->in->T, pool->in->d) != 0) {
        pthread_mutex_lock(&pool->mu);
        pool->failed = 1;
        pthread_mutex_unlock(&pool->mu);
        scratch_free(&w);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&pool->mu);
        int job = pool->next++;
        pthread_mutex_unlock(&pool->mu);
        if (job >= pool->njobs) break;
        double *dp = pool->dp_partial ? pool->dp_partial + (size_t)job * pool->in->d * pool->in->d : NULL;
        pool->run(pool->ctx, job, &w, dp);
    }
    scratch_free(&w);
    return NULL;
}

static int run_pool(pool_t *pool, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pool->njobs) nthreads = pool->njobs > 0 ? pool->njobs : 1;
    pthread_mutex_init(&pool->mu, NULL);
    pool->next = 0;
    pool->failed = 0;
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -1;
    int started = 0;
    for (int i = 0; i < nthreads; i++) {
        if (pthread_create(&th[i], NULL, worker, pool) == 0) started++;
        else break;
    }
    if (started == 0) worker(pool);
    for (int i = 0; i < started; i++) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&pool->mu);
    return pool->failed ? -1 : 0;
}

/* ------------------------------------------------------------------ forward */

typedef struct {
    const plx_in_t *in;
    double *out, *lse, *mu_k;
} fwd_ctx_t;

static void fwd_job(void *vctx, int job, scratch_t *w, double *unused) {
    (void)unused;
    fwd_ctx_t *ctx = (fwd_ctx_t *)vctx;
    const plx_in_t *in = ctx->in;
    const int b = job / in->H, h = job % in->H, d = in->d;
    for (int t = 0; t < in->T; t++) {
        double gbar;
        double L = forward_query(in, b, h, t, w, &gbar);
        size_t row = ((size_t)b * in->H + h) * in->T + t;
        if (ctx->lse) ctx->lse[row] = L;
        for (int j = 0; j < d; j++) {
            if (ctx->out) ctx->out[row * d + j] = w->o[j];
            if (ctx->mu_k) ctx->mu_k[row * d + j] = w->mu_k[j];
        }
    }
}

int plx_oracle_fwd(const double *q, const double *k, const double *v, const double *P,
                   int p_per_query, int B, int H, int T, int d,
                   double *out, double *lse, double *mu_k, int nthreads) {
    if (B < 1 || H < 1 || T < 1 || d < 1 || !q || !k || !v || !P) return 1;
    plx_in_t in = {q, k, v, P, NULL, B, H, T, d, p_per_query};
    fwd_ctx_t ctx = {&in, out, lse, mu_k};
    pool_t pool;
    memset(&pool, 0, sizeof(pool));
    pool.in = &in;
    pool.njobs = B * H;
    pool.run = fwd_job;
    pool.ctx = &ctx;
    return run_pool(&pool, nthreads) ? 2 : 0;
}

/* Forward at selected rows only: rows is n triples (b, h, t). */
typedef struct {
    const plx_in_t *in;
    const int64_t *rows;
    double *out, *lse, *mu_k;
} rows_ctx_t;

static void rows_job(void *vctx, int job, scratch_t *w, double *unused) {
    (void)unused;
    rows_ctx_t *ctx = (rows_ctx_t *)vctx;
    const int b = (int)ctx->rows[3 * job], h = (int)ctx->rows[3 * job + 1];
    const int t = (int)ctx->rows[3 * job + 2], d = ctx->in->d;
    double gbar;
    double L = forward_query(ctx->in, b, h, t, w, &gbar);
    if (ctx->lse) ctx->lse[job] = L;
    for (int j = 0; j < d; j++) {
        if (ctx->out) ctx->out[(size_t)job * d + j] = w->o[j];
        if (ctx->mu_k) ctx->mu_k[(size_t)job * d + j] = w->mu_k[j];
    }
}

int plx_oracle_fwd_rows(const double *q, const double *k, const double *v, const double *P,
                        int B, int H, int T, int d, const int64_t *rows, int n,
                        double *out, double *lse, double *mu_k, int nthreads) {
    if (B < 1 || H < 1 || T < 1 || d < 1 || n < 0 || !q || !k || !v || !P || (n && !rows)) return 1;
    for (int r = 0; r < n; r++) {
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= H ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= T)
            return 1;
    }
    plx_in_t in = {q, k, v, P, NULL, B, H, T, d, 0};
    rows_ctx_t ctx = {&in, rows, out, lse, mu_k};
    pool_t pool;
    memset(&pool, 0, sizeof(pool));
    pool.in = &in;
    pool.njobs = n;
    pool.run = rows_job;
    pool.ctx = &ctx;
    return run_pool(&pool, nthreads) ? 2 : 0;
}

/* ------------------------------------------------------- given probe (one pass)
 * The pages' literal form of the layer: the probe rho_t is given (in the paper
 * it comes from a learned projection of the layer input), not formed from
 * mu_k, and
 *   o_t = o^SA_t - Sigma_KV,t rho_t,
 *   Sigma_KV,t = sum_i p_ti (v_i - mu_v,t)(k_i - mu_k,t)^T   (reading: the
 *   softmax-weighted cross-covariance, centred at the softmax means).
 * rho is [B][H][T][d].  Written out term by term: the covariance applied to
 * rho is sum_i p_i (v_i - mu_v) ((k_i - mu_k) . rho). */
typedef struct {
    const plx_in_t *in;
    const double *rho;
    double *out, *lse;
} probe_ctx_t;

static double probe_query(const plx_in_t *in, const double *rho, int b, int h, int t, scratch_t *w) {
    const int d = in->d;
    const double c = 1.0 / sqrt((double)d);
    const double *Q = head_ptr(in->q, in, b, h);
    const double *K = head_ptr(in->k, in, b, h);
    const double *V = head_ptr(in->v, in, b, h);
    const double *qt = Q + (size_t)t * d;
    const double *rt = head_ptr(rho, in, b, h) + (size_t)t * d;

    double m = -INFINITY;
    for (int i = 0; i <= t; i++) {
        double acc = 0.0;
        for (int j = 0; j < d; j++) acc += qt[j] * K[(size_t)i * d + j];
        w->s[i] = c * acc;
        if (w->s[i] > m) m = w->s[i];
    }
    double Z = 0.0;
    for (int i = 0; i <= t; i++) Z += exp(w->s[i] - m);
    const double L = m + log(Z);
    for (int i = 0; i <= t; i++) w->p[i] = exp(w->s[i] - L);

    for (int j = 0; j < d; j++) { w->mu_v[j] = 0.0; w->mu_k[j] = 0.0; }
    for (int i = 0; i <= t; i++)
        for (int j = 0; j < d; j++) {
            w->mu_v[j] += w->p[i] * V[(size_t)i * d + j];
            w->mu_k[j] += w->p[i] * K[(size_t)i * d + j];
        }
    /* Sigma_KV rho = sum_i p_i (v_i - mu_v) ((k_i - mu_k) . rho) */
    for (int j = 0; j < d; j++) w->o[j] = 0.0;
    for (int i = 0; i <= t; i++) {
        double kr = 0.0;
        for (int j = 0; j < d; j++) kr += (K[(size_t)i * d + j] - w->mu_k[j]) * rt[j];
        for (int j = 0; j < d; j++) w->o[j] += w->p[i] * (V[(size_t)i * d + j] - w->mu_v[j]) * kr;
    }
    /* o = o^SA - Sigma_KV rho, with o^SA = mu_v */
    for (int j = 0; j < d; j++) w->o[j] = w->mu_v[j] - w->o[j];
    return L;
}

static void probe_job(void *vctx, int job, scratch_t *w, double *unused) {
    (void)unused;
    probe_ctx_t *ctx = (probe_ctx_t *)vctx;
    const plx_in_t *in = ctx->in;
    const int b = job / in->H, h = job % in->H, d = in->d;
    for (int t = 0; t < in->T; t++) {
        const double L = probe_query(in, ctx->rho, b, h, t, w);
        const size_t row = ((size_t)b * in->H + h) * in->T + t;
        if (ctx->lse) ctx->lse[row] = L;
        for (int j = 0; j < d; j++)
            if (ctx->out) ctx->out[row * d + j] = w->o[j];
    }
}

int plx_oracle_fwd_probe(const double *q, const double *k, const double *v, const double *rho, int B, int H,
                         int T, int d, double *out, double *lse, int nthreads) {
    if (B < 1 || H < 1 || T < 1 || d < 1 || !q || !k || !v || !rho) return 1;
    plx_in_t in = {q, k, v, NULL, NULL, B, H, T, d, 0};
    probe_ctx_t ctx = {&in, rho, out, lse};
    pool_t pool;
    memset(&pool, 0, sizeof(pool));
    pool.in = &in;
    pool.njobs = B * H;
    pool.run = probe_job;
    pool.ctx = &ctx;
    return run_pool(&pool, nthreads) ? 2 : 0;
}

/* The given-probe form at selected rows only: rows is n triples (b, h, t);
 * rho is still [B][H][T][d] (only the selected rows' probes are read). */
typedef struct {
    const plx_in_t *in;
    const double *rho;
    const int64_t *rows;
    double *out, *lse;
} probe_rows_ctx_t;

static void probe_rows_job(void *vctx, int job, scratch_t *w, double *unused) {
    (void)unused;
    probe_rows_ctx_t *ctx = (probe_rows_ctx_t *)vctx;
    const int b = (int)ctx->rows[3 * job], h = (int)ctx->rows[3 * job + 1];
    const int t = (int)ctx->rows[3 * job + 2], d = ctx->in->d;
    const double L = probe_query(ctx->in, ctx->rho, b, h, t, w);
    if (ctx->lse) ctx->lse[job] = L;
    for (int j = 0; j < d; j++)
        if (ctx->out) ctx->out[(size_t)job * d + j] = w->o[j];
}

int plx_oracle_fwd_probe_rows(const double *q, const double *k, const double *v, const double *rho, int B, int H,
                              int T, int d, const int64_t *rows, int n, double *out, double *lse, int nthreads) {
    if (B < 1 || H < 1 || T < 1 || d < 1 || n < 0 || !q || !k || !v || !rho || (n && !rows)) return 1;
    for (int r = 0; r < n; r++) {
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= H ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= T)
            return 1;
    }
    plx_in_t in = {q, k, v, NULL, NULL, B, H, T, d, 0};
    probe_rows_ctx_t ctx = {&in, rho, rows, out, lse};
    pool_t pool;
    memset(&pool, 0, sizeof(pool));
    pool.in = &in;
    pool.njobs = n;
    pool.run = probe_rows_job;
    pool.ctx = &ctx;
    return run_pool(&pool, nthreads) ? 2 : 0;
}

/* ----------------------------------------------------------------- backward */

typedef struct {
    const plx_in_t *in;
    const int32_t *heads; /* njobs pairs (b, h) */
    double *dq, *dk, *dv;
} bwd_ctx_t;

static void bwd_job(void *vctx, int job, scratch_t *w, double *dp) {
    bwd_ctx_t *ctx = (bwd_ctx_t *)vctx;
    const plx_in_t *in = ctx->in;
    const int b = ctx->heads[2 * job], h = ctx->heads[2 * job + 1];
    const int T = in->T, d = in->d;
    const double c = 1.0 / sqrt((double)d);
    const size_t base = ((size_t)b * in->H + h) * (size_t)T * d;
    const double *Q = in->q + base, *K = in->k + base, *V = in->v + base, *DO = in->dout + base;
    double *dq = ctx->dq + base, *dk = ctx->dk + base, *dv = ctx->dv + base;
    const double *P = in->P + (size_t)h * d * d;

    for (size_t j = 0; j < (size_t)T * d; j++) { dq[j] = 0.0; dk[j] = 0.0; dv[j] = 0.0; }
    for (int j = 0; j < d * d; j++) dp[j] = 0.0;

    for (int t = 0; t < T; t++) {
        double gbar;
        forward_query(in, b, h, t, w, &gbar);
        const double *dot = DO + (size_t)t * d;
        const double *qt = Q + (size_t)t * d;

        double ebar = 0.0;
        for (int i = 0; i <= t; i++) {
            double acc = 0.0;
            for (int j = 0; j < d; j++) acc += dot[j] * V[(size_t)i * d + j];
            w->e[i] = acc;
            ebar += w->p[i] * acc;
        }
        /* values and the g-branch */
        for (int j = 0; j < d; j++) w->du[j] = 0.0;
        for (int i = 0; i <= t; i++) {
            const double a = w->p[i] * (1.0 + w->g[i] - gbar);
            const double dg = w->p[i] * (w->e[i] - ebar);
            for (int j = 0; j < d; j++) {
                dv[(size_t)i * d + j] += a * dot[j];
                w->du[j] += dg * K[(size_t)i * d + j];
                dk[(size_t)i * d + j] += dg * w->u[j];
            }
        }
        /* projector and probe */
        for (int a = 0; a < d; a++)
            for (int bb = 0; bb < d; bb++) dp[(size_t)a * d + bb] += w->du[a] * w->delta[bb];
        for (int bb = 0; bb < d; bb++) {
            double acc = 0.0;
            for (int a = 0; a < d; a++) acc += P[(size_t)a * d + bb] * w->du[a];
            w->ddelta[bb] = acc;
        }
        for (int j = 0; j < d; j++) {
            dq[(size_t)t * d + j] += w->ddelta[j];
            w->dmu_k[j] = -w->ddelta[j];
        }
        for (int i = 0; i <= t; i++)
            for (int j = 0; j < d; j++) dk[(size_t)i * d + j] += w->p[i] * w->dmu_k[j];
        /* softmax weights */
        double doo = 0.0, mdm = 0.0;
        for (int j = 0; j < d; j++) { doo += dot[j] * w->o[j]; mdm += w->mu_k[j] * w->dmu_k[j]; }
        const double D = doo - gbar * ebar + mdm;
        for (int i = 0; i <= t; i++) {
            double kdm = 0.0;
            for (int j = 0; j < d; j++) kdm += K[(size_t)i * d + j] * w->dmu_k[j];
            const double ds = w->p[i] * (w->e[i] * (1.0 + w->g[i] - gbar) - w->g[i] * ebar + kdm - D);
            for (int j = 0; j < d; j++) {
                dq[(size_t)t * d + j] += c * ds * K[(size_t)i * d + j];
                dk[(size_t)i * d + j] += c * ds * qt[j];
            }
        }
    }
}

/* Gradients for the listed (b,h) heads.  dq/dk/dv are full [B][H][T][d]
 * arrays of which only the listed heads are written; dP[h] is the sum over
 * the listed heads with that h (in list order), other heads' dP are zeroed. */
int plx_oracle_bwd(const double *q, const double *k, const double *v, const double *P,
                   const double *dout, int B, int H, int T, int d,
                   const int32_t *heads, int nheads,
                   double *dq, double *dk, double *dv, double *dP, int nthreads) {
    if (B < 1 || H < 1 || T < 1 || d < 1 || nheads < 0 || !q || !k || !v || !P || !dout ||
        !dq || !dk || !dv || !dP || (nheads && !heads))
        return 1;
    for (int j = 0; j < nheads; j++)
        if (heads[2 * j] < 0 || heads[2 * j] >= B || heads[2 * j + 1] < 0 || heads[2 * j + 1] >= H)
            return 1;
    plx_in_t in = {q, k, v, P, dout, B, H, T, d, 0};
    bwd_ctx_t ctx = {&in, heads, dq, dk, dv};
    pool_t pool;
    memset(&pool, 0, sizeof(pool));
    pool.in = &in;
    pool.njobs = nheads;
    pool.run = bwd_job;
    pool.ctx = &ctx;
    pool.dp_partial = calloc((size_t)(nheads > 0 ? nheads : 1) * d * d, sizeof(double));
    if (!pool.dp_partial) return 2;
    int rc = run_pool(&pool, nthreads);
    for (size_t j = 0; j < (size_t)H * d * d; j++) dP[j] = 0.0;
    for (int job = 0; job < nheads; job++) {
        const int h = heads[2 * job + 1];
        for (int j = 0; j < d * d; j++) dP[(size_t)h * d * d + j] += pool.dp_partial[(size_t)job * d * d + j];
    }
    free(pool.dp_partial);
    return rc ? 2 : 0;
}
