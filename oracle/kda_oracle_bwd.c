/*
 * Gradient of the KDA recurrence: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE, like kda_oracle.c (same rules: only the tests, the
 * smoke check and bench.py's CPU legs load it; it shares nothing with the CUDA
 * kernels).
 *
 * The recurrence is the one of kda_oracle.c ("Kimi K3" study notes, section
 * 3-2 "2) Kimi Delta Attention"; "Kimi K3: 架构、训练与系统全景解析", section
 * 4.2.2), written per token as
 *
 *   X   = Diag(alpha) S_{t-1}          alpha = exp(log_alpha_t)
 *   p   = X^T k_t
 *   d   = beta_t (v_t - p)
 *   S_t = X + k_t d^T
 *   o_t = S_t^T q_t
 *
 * The pages print no gradient ("Kimi K3: 架构、训练与系统全景解析", section 7.1,
 * says the chunked kernel serves training as well as prefill, nothing more), so
 * this file is the chain rule applied to those five lines in reverse order,
 * token by token from the last one, for a loss whose gradients with respect to
 * every o_t (d_out) and the final state (d_final) are given:
 *
 *   dS  += q_t do_t^T                  (o_t = S_t^T q_t)
 *   dq_t = S_t do_t
 *   dd   = dS^T k_t,  dk_t = dS d      (S_t = X + k_t d^T, with dX = dS)
 *   dv_t = beta_t dd,  dbeta_t = dd . (v_t - p),  dp = -beta_t dd
 *   dX  = dS + k_t dp^T,  dk_t += X dp (p = X^T k_t)
 *   dlog_alpha_t[i] = sum_n dX[i][n] X[i][n],  dS_{t-1} = Diag(alpha) dX
 *
 * and d_init = dS_0.  The states S_{t-1} the reverse sweep needs are
 * recomputed from copies taken every kBlock tokens of a forward sweep (the
 * recomputation is the same forward arithmetic).
 *
 * Layouts as kda_oracle.c; gradients have the layout of their variables.
 * d_final and d_init may be NULL (zero / not written).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { kBlock = 64 };

typedef struct {
    const double *q, *k, *v, *log_alpha, *beta, *init_state, *d_out, *d_final;
    const int64_t *cu_seqlens;
    int64_t n_seqs, H, dk, dv;
    double *dq, *dk_, *dv_, *dla, *dbeta, *d_init;
    int64_t n_units, next_unit;
    pthread_mutex_t lock;
} bwd_job;

/* One forward token: S (in) -> X (written), p, d (written), S (out). */
static void step_fwd(int64_t dk, int64_t dv, const double *k, const double *v, const double *la,
                     double b, double *S, double *X, double *p, double *d) {
    for (int64_t i = 0; i < dk; ++i) {
        const double a = exp(la[i]);
        for (int64_t n = 0; n < dv; ++n) X[i * dv + n] = a * S[i * dv + n];
    }
    for (int64_t n = 0; n < dv; ++n) p[n] = 0.0;
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t n = 0; n < dv; ++n) p[n] += k[i] * X[i * dv + n];
    for (int64_t n = 0; n < dv; ++n) d[n] = b * (v[n] - p[n]);
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t n = 0; n < dv; ++n) S[i * dv + n] = X[i * dv + n] + k[i] * d[n];
}

typedef struct {
    double *ckpt;    /* state before every kBlock-th token of the chain */
    double *X, *P, *Dl; /* X, p, d of the tokens of one block */
    double *S, *dS, *dX, *tmp;
} bwd_scratch;

static void run_chain(const bwd_job *j, int64_t seq, int64_t h, bwd_scratch *w) {
    const int64_t H = j->H, dk = j->dk, dv = j->dv, m = dk * dv;
    const int64_t t0 = j->cu_seqlens[seq], t1 = j->cu_seqlens[seq + 1], len = t1 - t0;
    const int64_t nb = (len + kBlock - 1) / kBlock;
#define ROW(ptr, t, width) ((ptr) + ((t) * H + h) * (width))
    /* forward sweep: the state before each block */
    if (j->init_state) memcpy(w->S, j->init_state + (seq * H + h) * m, sizeof(double) * m);
    else memset(w->S, 0, sizeof(double) * m);
    for (int64_t t = t0; t < t1; ++t) {
        if ((t - t0) % kBlock == 0) memcpy(w->ckpt + ((t - t0) / kBlock) * m, w->S, sizeof(double) * m);
        step_fwd(dk, dv, ROW(j->k, t, dk), ROW(j->v, t, dv), ROW(j->log_alpha, t, dk),
                 j->beta[t * H + h], w->S, w->X, w->P, w->Dl);
    }
    /* reverse sweep */
    if (j->d_final) memcpy(w->dS, j->d_final + (seq * H + h) * m, sizeof(double) * m);
    else memset(w->dS, 0, sizeof(double) * m);
    for (int64_t blk = nb - 1; blk >= 0; --blk) {
        const int64_t a = t0 + blk * kBlock, e = a + kBlock < t1 ? a + kBlock : t1;
        memcpy(w->S, w->ckpt + blk * m, sizeof(double) * m);
        for (int64_t t = a; t < e; ++t)
            step_fwd(dk, dv, ROW(j->k, t, dk), ROW(j->v, t, dv), ROW(j->log_alpha, t, dk),
                     j->beta[t * H + h], w->S, w->X + (t - a) * m, w->P + (t - a) * dv,
                     w->Dl + (t - a) * dv);
        for (int64_t t = e - 1; t >= a; --t) {
            const double *X = w->X + (t - a) * m, *p = w->P + (t - a) * dv;
            const double *d = w->Dl + (t - a) * dv;
            const double *q = ROW(j->q, t, dk), *k = ROW(j->k, t, dk), *v = ROW(j->v, t, dv);
            const double *la = ROW(j->log_alpha, t, dk), *dout = ROW(j->d_out, t, dv);
            const double b = j->beta[t * H + h];
            double *dq = ROW(j->dq, t, dk), *dkk = ROW(j->dk_, t, dk), *dvv = ROW(j->dv_, t, dv);
            double *dla = ROW(j->dla, t, dk);
            /* o_t = S_t^T q: dS += q do^T, dq = S_t do with S_t = X + k d^T */
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t n = 0; n < dv; ++n) w->dS[i * dv + n] += q[i] * dout[n];
            for (int64_t i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int64_t n = 0; n < dv; ++n) acc += (X[i * dv + n] + k[i] * d[n]) * dout[n];
                dq[i] = acc;
            }
            /* S_t = X + k d^T: dd = dS^T k, dk = dS d */
            double *dd = w->tmp;
            for (int64_t n = 0; n < dv; ++n) dd[n] = 0.0;
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t n = 0; n < dv; ++n) dd[n] += w->dS[i * dv + n] * k[i];
            for (int64_t i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int64_t n = 0; n < dv; ++n) acc += w->dS[i * dv + n] * d[n];
                dkk[i] = acc;
            }
            /* d = beta (v - p) */
            double db = 0.0;
            for (int64_t n = 0; n < dv; ++n) {
                dvv[n] = b * dd[n];
                db += dd[n] * (v[n] - p[n]);
            }
            j->dbeta[t * H + h] = db;
            /* p = X^T k, with dp = -beta dd: dX = dS + k dp^T, dk += X dp */
            for (int64_t i = 0; i < dk; ++i) {
                double acc = 0.0, la_acc = 0.0;
                for (int64_t n = 0; n < dv; ++n) {
                    const double dp = -b * dd[n];
                    const double dx = w->dS[i * dv + n] + k[i] * dp;
                    acc += X[i * dv + n] * dp;
                    la_acc += dx * X[i * dv + n];
                    w->dX[i * dv + n] = dx;
                }
                dkk[i] += acc;
                /* X = Diag(exp(log_alpha)) S_{t-1} */
                dla[i] = la_acc;
                const double al = exp(la[i]);
                for (int64_t n = 0; n < dv; ++n) w->dS[i * dv + n] = al * w->dX[i * dv + n];
            }
        }
    }
    if (j->d_init) memcpy(j->d_init + (seq * H + h) * m, w->dS, sizeof(double) * m);
#undef ROW
}

static void *bwd_worker(void *arg) {
    bwd_job *job = (bwd_job *)arg;
    const int64_t m = job->dk * job->dv;
    int64_t max_len = 0;
    for (int64_t s = 0; s < job->n_seqs; ++s) {
        const int64_t l = job->cu_seqlens[s + 1] - job->cu_seqlens[s];
        if (l > max_len) max_len = l;
    }
    const int64_t n_ck = (max_len + kBlock - 1) / kBlock + 1;
    bwd_scratch w;
    w.ckpt = (double *)malloc(sizeof(double) * m * n_ck);
    w.X = (double *)malloc(sizeof(double) * m * kBlock);
    w.P = (double *)malloc(sizeof(double) * job->dv * kBlock);
    w.Dl = (double *)malloc(sizeof(double) * job->dv * kBlock);
    w.S = (double *)malloc(sizeof(double) * m);
    w.dS = (double *)malloc(sizeof(double) * m);
    w.dX = (double *)malloc(sizeof(double) * m);
    w.tmp = (double *)malloc(sizeof(double) * job->dv);
    void *rc = NULL;
    if (!w.ckpt || !w.X || !w.P || !w.Dl || !w.S || !w.dS || !w.dX || !w.tmp) {
        rc = (void *)1;
    } else {
        for (;;) {
            pthread_mutex_lock(&job->lock);
            const int64_t u = job->next_unit++;
            pthread_mutex_unlock(&job->lock);
            if (u >= job->n_units) break;
            run_chain(job, u / job->H, u % job->H, &w);
        }
    }
    free(w.ckpt); free(w.X); free(w.P); free(w.Dl); free(w.S); free(w.dS); free(w.dX); free(w.tmp);
    return rc;
}

/* Returns 0 on success, 1 on bad arguments, 2 on allocation / thread failure. */
int kda_oracle_chunk_bwd(const double *q, const double *k, const double *v,
                         const double *log_alpha, const double *beta, const double *init_state,
                         const int64_t *cu_seqlens, int64_t n_seqs, int64_t H, int64_t dk,
                         int64_t dv, const double *d_out, const double *d_final, double *dq,
                         double *dk_, double *dv_, double *dla, double *dbeta, double *d_init,
                         int n_threads) {
    if (!cu_seqlens || n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    if (cu_seqlens[0] != 0) return 1;
    for (int64_t s = 0; s < n_seqs; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return 1;
    if (cu_seqlens[n_seqs] > 0 && (!q || !k || !v || !log_alpha || !beta || !d_out || !dq ||
                                   !dk_ || !dv_ || !dla || !dbeta))
        return 1;
    bwd_job job;
    job.q = q; job.k = k; job.v = v; job.log_alpha = log_alpha; job.beta = beta;
    job.init_state = init_state; job.d_out = d_out; job.d_final = d_final;
    job.cu_seqlens = cu_seqlens; job.n_seqs = n_seqs; job.H = H; job.dk = dk; job.dv = dv;
    job.dq = dq; job.dk_ = dk_; job.dv_ = dv_; job.dla = dla; job.dbeta = dbeta;
    job.d_init = d_init;
    job.n_units = n_seqs * H;
    job.next_unit = 0;
    pthread_mutex_init(&job.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > job.n_units) n_threads = (int)(job.n_units > 0 ? job.n_units : 1);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!tids) return 2;
    int started = 0, rc = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&tids[i], NULL, bwd_worker, &job) != 0) { rc = 2; break; }
        ++started;
    }
    if (started == 0) rc = bwd_worker(&job) != NULL ? 2 : 0;
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tids[i], &ret);
        if (ret != NULL) rc = 2;
    }
    free(tids);
    pthread_mutex_destroy(&job.lock);
    return rc;
}
