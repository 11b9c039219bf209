/*
 * KDA recurrence oracle: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check in __graft_entry__ and
 * the CPU-baseline leg of bench.py load this library.  The product path
 * (gated_delta_rule_13_gb300/) never links, loads or calls it, and it shares
 * no code, header or constant with the CUDA kernels.
 *
 * What it computes, token by token for every (sequence, head):
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T q_t
 *
 * with S in R^{dk x dv}, alpha_t = exp(log_alpha_t) per key channel, and the
 * read-out taken from the post-update state with no scale factor.
 * Sources: "Kimi K3" study notes (dimensionstp), section 3-2 "2) Kimi Delta
 * Attention", state-update and read-out equations; "Kimi K3: 架构、训练与系统
 * 全景解析", section 4.2.2 (three-part reading of the update: per-channel decay,
 * erase along k_t, write beta_t k_t v_t^T; read-out S_t^T q_t); "AI-Workshop
 * 文献分享 #15", section 7.2 (S_t in R^{dk x dv}, rows = key address space).
 *
 * The product (I - beta k k^T) X with X = Diag(alpha) S is evaluated as
 * X - beta k (k^T X): the same matrix, associativity only, so that a token
 * costs O(dk dv) instead of O(dk^2 dv).  No chunking, blocking or reordering
 * beyond that.
 *
 * Layouts (row-major, packed varlen, token-major):
 *   q, k, log_alpha : [n_tokens, H, dk]      v, out : [n_tokens, H, dv]
 *   beta            : [n_tokens, H]
 *   init_state, final_state : [n_seqs, H, dk, dv]   (dv contiguous)
 *   cu_seqlens      : [n_seqs + 1], cu_seqlens[0] = 0, non-decreasing
 * init_state may be NULL (zero state).  final_state may be NULL.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *log_alpha, *beta, *init_state;
    const int64_t *cu_seqlens;
    int64_t n_seqs, H, dk, dv;
    double *out, *final_state;
    int64_t n_units;
    int64_t next_unit; /* shared work counter */
    pthread_mutex_t lock;
} fwd_job;

static int64_t take_unit(fwd_job *job) {
    pthread_mutex_lock(&job->lock);
    int64_t u = job->next_unit++;
    pthread_mutex_unlock(&job->lock);
    return u;
}

/* One (sequence, head) chain of the recurrence. */
static void run_chain(const fwd_job *j, int64_t seq, int64_t h, double *S, double *tmp) {
    const int64_t H = j->H, dk = j->dk, dv = j->dv;
    const int64_t t0 = j->cu_seqlens[seq], t1 = j->cu_seqlens[seq + 1];

    if (j->init_state) {
        memcpy(S, j->init_state + (seq * H + h) * dk * dv, sizeof(double) * dk * dv);
    } else {
        memset(S, 0, sizeof(double) * dk * dv);
    }
    for (int64_t t = t0; t < t1; ++t) {
        const double *qt = j->q + (t * H + h) * dk;
        const double *kt = j->k + (t * H + h) * dk;
        const double *vt = j->v + (t * H + h) * dv;
        const double *lat = j->log_alpha + (t * H + h) * dk;
        const double bt = j->beta[t * H + h];

        /* X = Diag(alpha_t) S_{t-1}: key channel i keeps alpha_{t,i} of row i. */
        for (int64_t i = 0; i < dk; ++i) {
            const double a = exp(lat[i]);
            for (int64_t n = 0; n < dv; ++n) S[i * dv + n] *= a;
        }
        /* tmp = k_t^T X  (what the decayed state returns for address k_t). */
        for (int64_t n = 0; n < dv; ++n) tmp[n] = 0.0;
        for (int64_t i = 0; i < dk; ++i) {
            const double ki = kt[i];
            for (int64_t n = 0; n < dv; ++n) tmp[n] += ki * S[i * dv + n];
        }
        /* S_t = X - beta k (k^T X) + beta k v^T = X + beta k (v - k^T X)^T. */
        for (int64_t n = 0; n < dv; ++n) tmp[n] = bt * (vt[n] - tmp[n]);
        for (int64_t i = 0; i < dk; ++i) {
            const double ki = kt[i];
            for (int64_t n = 0; n < dv; ++n) S[i * dv + n] += ki * tmp[n];
        }
        /* o_t = S_t^T q_t. */
        double *ot = j->out + (t * H + h) * dv;
        for (int64_t n = 0; n < dv; ++n) ot[n] = 0.0;
        for (int64_t i = 0; i < dk; ++i) {
            const double qi = qt[i];
            for (int64_t n = 0; n < dv; ++n) ot[n] += qi * S[i * dv + n];
        }
    }
    if (j->final_state) {
        memcpy(j->final_state + (seq * H + h) * dk * dv, S, sizeof(double) * dk * dv);
    }
}

static void *fwd_worker(void *arg) {
    fwd_job *job = (fwd_job *)arg;
    double *S = (double *)malloc(sizeof(double) * job->dk * job->dv);
    double *tmp = (double *)malloc(sizeof(double) * job->dv);
    if (!S || !tmp) {
        free(S);
        free(tmp);
        return (void *)1;
    }
    for (;;) {
        const int64_t u = take_unit(job);
        if (u >= job->n_units) break;
        run_chain(job, u / job->H, u % job->H, S, tmp);
    }
    free(S);
    free(tmp);
    return NULL;
}

/* Returns 0 on success, 1 on bad arguments, 2 on allocation / thread failure. */
int kda_oracle_chunk_fwd(const double *q, const double *k, const double *v,
                         const double *log_alpha, const double *beta,
                         const double *init_state, const int64_t *cu_seqlens,
                         int64_t n_seqs, int64_t H, int64_t dk, int64_t dv,
                         double *out, double *final_state, int n_threads) {
    if (!cu_seqlens || n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    if (cu_seqlens[0] != 0) return 1;
    for (int64_t s = 0; s < n_seqs; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return 1;
    if (cu_seqlens[n_seqs] > 0 && (!q || !k || !v || !log_alpha || !beta || !out)) return 1;

    fwd_job job;
    job.q = q; job.k = k; job.v = v; job.log_alpha = log_alpha; job.beta = beta;
    job.init_state = init_state; job.cu_seqlens = cu_seqlens;
    job.n_seqs = n_seqs; job.H = H; job.dk = dk; job.dv = dv;
    job.out = out; job.final_state = final_state;
    job.n_units = n_seqs * H;
    job.next_unit = 0;
    pthread_mutex_init(&job.lock, NULL);

    if (n_threads < 1) n_threads = 1;
    if (n_threads > job.n_units) n_threads = (int)(job.n_units > 0 ? job.n_units : 1);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!tids) return 2;
    int started = 0, rc = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&tids[i], NULL, fwd_worker, &job) != 0) { rc = 2; break; }
        ++started;
    }
    if (started == 0) { /* run inline if no thread could start */
        if (fwd_worker(&job) != NULL) rc = 2; else rc = 0;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tids[i], &ret);
        if (ret != NULL) rc = 2;
    }
    free(tids);
    pthread_mutex_destroy(&job.lock);
    return rc;
}

/*
 * One recurrent decode step for B independent sequences x H heads, state
 * updated in place (the state advances in place during decoding: "Kimi K3:
 * 架构、训练与系统全景解析" section 4.2.7).  Same update and read-out as above.
 *   state : [B, H, dk, dv]   q, k, log_alpha : [B, H, dk]   v, out : [B, H, dv]
 *   beta  : [B, H]
 * Single-threaded: a step is O(B H dk dv).
 */
int kda_oracle_decode_step(double *state, const double *q, const double *k, const double *v,
                           const double *log_alpha, const double *beta,
                           int64_t B, int64_t H, int64_t dk, int64_t dv, double *out) {
    if (!state || !q || !k || !v || !log_alpha || !beta || !out) return 1;
    if (B < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    double *p = (double *)malloc(sizeof(double) * dv);
    if (!p) return 2;
    for (int64_t u = 0; u < B * H; ++u) {
        double *S = state + u * dk * dv;
        const double *qt = q + u * dk, *kt = k + u * dk, *vt = v + u * dv;
        const double *lat = log_alpha + u * dk;
        const double bt = beta[u];
        for (int64_t i = 0; i < dk; ++i) {
            const double a = exp(lat[i]);
            for (int64_t n = 0; n < dv; ++n) S[i * dv + n] *= a;
        }
        for (int64_t n = 0; n < dv; ++n) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += kt[i] * S[i * dv + n];
            p[n] = bt * (vt[n] - acc);
        }
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t n = 0; n < dv; ++n) S[i * dv + n] += kt[i] * p[n];
        for (int64_t n = 0; n < dv; ++n) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += qt[i] * S[i * dv + n];
            out[u * dv + n] = acc;
        }
    }
    free(p);
    return 0;
}
