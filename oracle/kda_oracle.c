/*
 * kda_oracle.c -- plain fp64 CPU oracle for the Kimi Delta Attention (KDA)
 * recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The CUDA product
 * path never calls it and shares no code, header or table with it.
 *
 * What it computes, per sequence n and head h, token by token, in fp64:
 *
 *   alpha_t = exp(g_t)                        (per key channel)
 *   M       = Diag(alpha_t) S_{t-1}           decay the rows (key channels)
 *   p       = M^T k_t                         what the memory returns for k_t
 *   u       = beta_t (v_t - p)                the correction
 *   S_t     = M + k_t u^T                     write
 *   o_t     = S_t^T q_t                       read, after the write
 *
 * Sources (the pages describe one recurrence in several equivalent forms):
 *  - "Understanding Kimi K3's Attention" (dhruvpendharkar.github.io): the
 *    state-update equation S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1}
 *    + beta_t k_t v_t^T, the readout equation o_t = S_t^T q_t, and the
 *    rewritten "delta" form S_t = Diag(alpha_t)S_{t-1} + beta_t k_t (v_t -
 *    (Diag(alpha_t)S_{t-1})^T k_t)^T that this loop follows.  The symbol
 *    table gives alpha_t = exp(g_t) per channel and beta_t in (0,1); the
 *    log-decay bound equation gives g_t in (g_min, 0) with g_min = -5.
 *  - "Hybrid Attention" (kimi-k3.adriaflores.com), section "KDA: don't
 *    write the same information twice": retain (S = alpha*S, alpha
 *    broadcast over the value axis, i.e. it scales key channels), predict
 *    v_old = S^T k, correct by beta*(v - v_old), and the query reads the
 *    updated S.
 *  - "Kimi K3 course, lesson 2: KDA: the memory matrix": the read uses S at
 *    time t, not t-1.
 *
 * Layouts (row-major, contiguous, fp64):
 *   q, k  [T_tot, H, d_k];  v, out [T_tot, H, d_v];  g [T_tot, H, d_k];
 *   beta  [T_tot, H];       states [N, H, d_k, d_v] (row i = key channel i).
 *   cu_seqlens int32 [N+1]: sequence n covers tokens [cu[n], cu[n+1]).
 *
 * Domain: g must lie in [-5, 0] and beta in [0, 1] (the pages' open
 * intervals, closed so that the special cases beta = 0, beta = 1 and
 * alpha = 1 are inside).  Out-of-domain input returns -1 before any work.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include "kda_oracle.h"

#define KDA_ORACLE_G_MIN (-5.0)

typedef struct {
    int64_t h_count, dk, dv;
    const double *q, *k, *v, *g, *beta, *init_state;
    const int32_t *cu;
    double *out, *final_state;
    int64_t n_items;
    int64_t next; /* work counter, guarded by lock */
    pthread_mutex_t lock;
} oracle_job;

/* One (sequence, head) pair: the token loop written out. */
static void run_one(const oracle_job *J, int64_t n, int64_t h, double *S,
                    double *alpha, double *p, double *u) {
    const int64_t H = J->h_count, dk = J->dk, dv = J->dv;
    if (J->init_state)
        memcpy(S, J->init_state + (n * H + h) * dk * dv, sizeof(double) * dk * dv);
    else
        memset(S, 0, sizeof(double) * dk * dv);

    for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
        const double *qt = J->q + (t * H + h) * dk;
        const double *kt = J->k + (t * H + h) * dk;
        const double *vt = J->v + (t * H + h) * dv;
        const double *gt = J->g + (t * H + h) * dk;
        const double bt = J->beta[t * H + h];
        double *ot = J->out + (t * H + h) * dv;

        for (int64_t i = 0; i < dk; ++i) alpha[i] = exp(gt[i]);
        /* M = Diag(alpha) S */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= alpha[i];
        /* p = M^T k */
        for (int64_t j = 0; j < dv; ++j) p[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) p[j] += S[i * dv + j] * kt[i];
        /* u = beta (v - p) */
        for (int64_t j = 0; j < dv; ++j) u[j] = bt * (vt[j] - p[j]);
        /* S = M + k u^T */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * u[j];
        /* o = S^T q */
        for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) ot[j] += S[i * dv + j] * qt[i];
    }
    if (J->final_state)
        memcpy(J->final_state + (n * H + h) * dk * dv, S, sizeof(double) * dk * dv);
}

static void *worker(void *arg) {
    oracle_job *J = (oracle_job *)arg;
    const int64_t dk = J->dk, dv = J->dv;
    double *S = (double *)malloc(sizeof(double) * dk * dv);
    double *alpha = (double *)malloc(sizeof(double) * dk);
    double *p = (double *)malloc(sizeof(double) * dv);
    double *u = (double *)malloc(sizeof(double) * dv);
    if (!S || !alpha || !p || !u) {
        free(S); free(alpha); free(p); free(u);
        return (void *)1;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t item = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (item >= J->n_items) break;
        run_one(J, item / J->h_count, item % J->h_count, S, alpha, p, u);
    }
    free(S); free(alpha); free(p); free(u);
    return NULL;
}

int kda_oracle_num_cpus(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

int kda_oracle_prefill(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                       int32_t d_k, int32_t d_v, const double *q, const double *k,
                       const double *v, const double *g, const double *beta,
                       const double *init_state, const int32_t *cu_seqlens,
                       double *out, double *final_state, int32_t num_threads) {
    if (num_seqs < 0 || total_tokens < 0 || num_heads <= 0 || d_k <= 0 || d_v <= 0)
        return -1;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return -1;

    int32_t *cu_local = NULL;
    const int32_t *cu = cu_seqlens;
    if (!cu) {
        if (num_seqs == 0 ? total_tokens != 0 : total_tokens % num_seqs != 0) return -1;
        cu_local = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_seqs + 1));
        if (!cu_local) return -1;
        int32_t len = num_seqs ? total_tokens / num_seqs : 0;
        for (int32_t n = 0; n <= num_seqs; ++n) cu_local[n] = n * len;
        cu = cu_local;
    }
    int rc = 0;
    if (cu[0] != 0 || cu[num_seqs] != total_tokens) rc = -1;
    for (int32_t n = 0; n < num_seqs && rc == 0; ++n)
        if (cu[n + 1] < cu[n]) rc = -1;
    /* domain of the gates */
    const int64_t nk = (int64_t)total_tokens * num_heads * d_k;
    for (int64_t i = 0; i < nk && rc == 0; ++i)
        if (!(g[i] >= KDA_ORACLE_G_MIN && g[i] <= 0.0)) rc = -1;
    for (int64_t i = 0; i < (int64_t)total_tokens * num_heads && rc == 0; ++i)
        if (!(beta[i] >= 0.0 && beta[i] <= 1.0)) rc = -1;
    if (rc != 0) {
        free(cu_local);
        return rc;
    }

    oracle_job J;
    J.h_count = num_heads; J.dk = d_k; J.dv = d_v;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.init_state = init_state;
    J.cu = cu; J.out = out; J.final_state = final_state;
    J.n_items = (int64_t)num_seqs * num_heads;
    J.next = 0;
    pthread_mutex_init(&J.lock, NULL);

    int nt = num_threads > 0 ? num_threads : kda_oracle_num_cpus();
    if (nt > J.n_items) nt = (int)(J.n_items > 0 ? J.n_items : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    int started = 0;
    if (th) {
        for (int i = 1; i < nt; ++i)
            if (pthread_create(&th[i], NULL, worker, &J) == 0) ++started;
            else break;
    }
    if (worker(&J) != NULL) rc = -1;
    for (int i = 1; i <= started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -1;
    }
    free(th);
    pthread_mutex_destroy(&J.lock);
    free(cu_local);
    return rc;
}

/* Gradients of the recurrence, reverse mode, token by token (the pages'
 * training path compares the chunked computation's gradients with those of
 * the simple recurrent version: "Hybrid Attention", section "But isn't a
 * recurrent update sequential?").  For a loss L with dL/do_t = d_out[t] and
 * dL/dS_T = d_final_state (NULL => 0), per (sequence, head), the forward
 * states S_0..S_T are kept; then for t = T..1, with dS = dL/dS_t:
 *
 *   dS   += q_t do_t^T,  dq_t = S_t do_t                    (o_t = S_t^T q_t)
 *   du    = dS^T k_t,    dk_t = dS u_t                      (S_t = M_t + k_t u_t^T)
 *   dv_t  = beta_t du,   dbeta_t = du . (v_t - p_t),  dp = -beta_t du
 *   dM    = dS + k_t dp^T,  dk_t += M_t dp                   (p_t = M_t^T k_t)
 *   dg_t[i] = alpha_t[i] sum_j dM[i][j] S_{t-1}[i][j],  dS <- Diag(alpha_t) dM
 *                                                            (M_t = Diag(alpha_t) S_{t-1})
 *
 * and dL/dS_0 is the dS left after t = 1. */
typedef struct {
    int64_t h_count, dk, dv;
    const double *q, *k, *v, *g, *beta, *init_state, *d_out, *d_final;
    const int32_t *cu;
    double *dq, *dkk, *dvv, *dg, *dbeta, *d_init;
    int64_t n_items, next;
    pthread_mutex_t lock;
} oracle_bwd_job;

static int bwd_one(const oracle_bwd_job *J, int64_t n, int64_t h) {
    const int64_t H = J->h_count, dk = J->dk, dv = J->dv, sz = dk * dv;
    const int64_t a = J->cu[n], L = J->cu[n + 1] - J->cu[n];
    double *st = (double *)malloc(sizeof(double) * (size_t)((L + 1) * sz));
    double *dS = (double *)malloc(sizeof(double) * (size_t)sz);
    double *dM = (double *)malloc(sizeof(double) * (size_t)sz);
    double *w = (double *)malloc(sizeof(double) * (size_t)(dk + 4 * dv));
    if (!st || !dS || !dM || !w) {
        free(st); free(dS); free(dM); free(w);
        return -1;
    }
    double *al = w, *pp = w + dk, *uu = pp + dv, *du = uu + dv, *dp = du + dv;
    if (J->init_state) memcpy(st, J->init_state + (n * H + h) * sz, sizeof(double) * sz);
    else memset(st, 0, sizeof(double) * sz);
    /* forward, keeping every state */
    for (int64_t t = 0; t < L; ++t) {
        const int64_t ix = (a + t) * H + h;
        const double *kt = J->k + ix * dk, *vt = J->v + ix * dv, *gt = J->g + ix * dk;
        const double *S0 = st + t * sz;
        double *S1 = st + (t + 1) * sz;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S1[i * dv + j] = exp(gt[i]) * S0[i * dv + j];
        for (int64_t j = 0; j < dv; ++j) pp[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) pp[j] += S1[i * dv + j] * kt[i];
        for (int64_t j = 0; j < dv; ++j) uu[j] = J->beta[ix] * (vt[j] - pp[j]);
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S1[i * dv + j] += kt[i] * uu[j];
    }
    /* backward */
    if (J->d_final) memcpy(dS, J->d_final + (n * H + h) * sz, sizeof(double) * sz);
    else memset(dS, 0, sizeof(double) * sz);
    for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t ix = (a + t) * H + h;
        const double *qt = J->q + ix * dk, *kt = J->k + ix * dk, *vt = J->v + ix * dv;
        const double *gt = J->g + ix * dk, *dot = J->d_out + ix * dv;
        const double bt = J->beta[ix];
        const double *Sp = st + t * sz, *St = st + (t + 1) * sz;
        double *dqt = J->dq + ix * dk, *dkt = J->dkk + ix * dk, *dgt = J->dg + ix * dk;
        double *dvt = J->dvv + ix * dv;
        for (int64_t i = 0; i < dk; ++i) al[i] = exp(gt[i]);
        /* o_t = S_t^T q_t */
        for (int64_t i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                dS[i * dv + j] += qt[i] * dot[j];
                acc += St[i * dv + j] * dot[j];
            }
            dqt[i] = acc;
        }
        /* recompute p_t and u_t from M_t = Diag(alpha) S_{t-1} */
        for (int64_t j = 0; j < dv; ++j) pp[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) pp[j] += al[i] * Sp[i * dv + j] * kt[i];
        for (int64_t j = 0; j < dv; ++j) uu[j] = bt * (vt[j] - pp[j]);
        /* S_t = M_t + k u^T */
        for (int64_t j = 0; j < dv; ++j) du[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                du[j] += dS[i * dv + j] * kt[i];
                acc += dS[i * dv + j] * uu[j];
            }
            dkt[i] = acc;
        }
        /* u = beta (v - p) */
        double db = 0.0;
        for (int64_t j = 0; j < dv; ++j) {
            dvt[j] = bt * du[j];
            db += du[j] * (vt[j] - pp[j]);
            dp[j] = -bt * du[j];
        }
        J->dbeta[ix] = db;
        /* p = M^T k and M = Diag(alpha) S_{t-1} */
        for (int64_t i = 0; i < dk; ++i) {
            double acc = 0.0, ga = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                dM[i * dv + j] = dS[i * dv + j] + kt[i] * dp[j];
                acc += al[i] * Sp[i * dv + j] * dp[j];
                ga += dM[i * dv + j] * Sp[i * dv + j];
            }
            dkt[i] += acc;
            dgt[i] = al[i] * ga;
            for (int64_t j = 0; j < dv; ++j) dS[i * dv + j] = al[i] * dM[i * dv + j];
        }
    }
    memcpy(J->d_init + (n * H + h) * sz, dS, sizeof(double) * sz);
    free(st); free(dS); free(dM); free(w);
    return 0;
}

static void *bwd_worker(void *arg) {
    oracle_bwd_job *J = (oracle_bwd_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t item = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (item >= J->n_items) break;
        if (bwd_one(J, item / J->h_count, item % J->h_count) != 0) return (void *)1;
    }
    return NULL;
}

int kda_oracle_backward(int32_t num_seqs, int32_t total_tokens, int32_t num_heads, int32_t d_k,
                        int32_t d_v, const double *q, const double *k, const double *v,
                        const double *g, const double *beta, const double *init_state,
                        const int32_t *cu_seqlens, const double *d_out,
                        const double *d_final_state, double *dq, double *dk, double *dv,
                        double *dg, double *dbeta, double *d_init_state, int32_t num_threads) {
    if (num_seqs < 0 || total_tokens < 0 || num_heads <= 0 || d_k <= 0 || d_v <= 0) return -1;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !d_out || !dq || !dk || !dv ||
                             !dg || !dbeta))
        return -1;
    if (num_seqs > 0 && !d_init_state) return -1;
    int32_t *cu_local = NULL;
    const int32_t *cu = cu_seqlens;
    if (!cu) {
        if (num_seqs == 0 ? total_tokens != 0 : total_tokens % num_seqs != 0) return -1;
        cu_local = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_seqs + 1));
        if (!cu_local) return -1;
        const int32_t len = num_seqs ? total_tokens / num_seqs : 0;
        for (int32_t n = 0; n <= num_seqs; ++n) cu_local[n] = n * len;
        cu = cu_local;
    }
    int rc = 0;
    if (cu[0] != 0 || cu[num_seqs] != total_tokens) rc = -1;
    for (int32_t n = 0; n < num_seqs && rc == 0; ++n)
        if (cu[n + 1] < cu[n]) rc = -1;
    for (int64_t i = 0; i < (int64_t)total_tokens * num_heads * d_k && rc == 0; ++i)
        if (!(g[i] >= KDA_ORACLE_G_MIN && g[i] <= 0.0)) rc = -1;
    for (int64_t i = 0; i < (int64_t)total_tokens * num_heads && rc == 0; ++i)
        if (!(beta[i] >= 0.0 && beta[i] <= 1.0)) rc = -1;
    if (rc != 0) {
        free(cu_local);
        return rc;
    }
    oracle_bwd_job J;
    J.h_count = num_heads; J.dk = d_k; J.dv = d_v;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.init_state = init_state;
    J.d_out = d_out; J.d_final = d_final_state; J.cu = cu;
    J.dq = dq; J.dkk = dk; J.dvv = dv; J.dg = dg; J.dbeta = dbeta; J.d_init = d_init_state;
    J.n_items = (int64_t)num_seqs * num_heads;
    J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    int nt = num_threads > 0 ? num_threads : kda_oracle_num_cpus();
    if (nt > J.n_items) nt = (int)(J.n_items > 0 ? J.n_items : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    int started = 0;
    if (th) {
        for (int i = 1; i < nt; ++i) {
            if (pthread_create(&th[i], NULL, bwd_worker, &J) == 0) ++started;
            else break;
        }
    }
    if (bwd_worker(&J) != NULL) rc = -1;
    for (int i = 1; i <= started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -1;
    }
    free(th);
    pthread_mutex_destroy(&J.lock);
    free(cu_local);
    return rc;
}

/* Gated DeltaNet and the delta rule ("Kimi K3.1 and the Road From Softmax
 * Attention to Kimi Delta Attention", sections "3. The delta rule" and "4.
 * Gating"): S_t = (I - beta_t k_t k_t^T) alpha_t S_{t-1} + beta_t k_t v_t^T
 * with one decay alpha_t = exp(g_head[t,h]) per head and step; with g_head
 * NULL, alpha_t = 1, the delta rule.  A scalar decay scales every key channel
 * alike, so this is the channel-wise recurrence above with g[t,h,c] =
 * g_head[t,h] for every channel c. */
int kda_oracle_prefill_scalar_decay(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                    int32_t d_k, int32_t d_v, const double *q, const double *k,
                                    const double *v, const double *g_head, const double *beta,
                                    const double *init_state, const int32_t *cu_seqlens,
                                    double *out, double *final_state, int32_t num_threads) {
    if (total_tokens < 0 || num_heads <= 0 || d_k <= 0) return -1;
    const int64_t n = (int64_t)total_tokens * num_heads * d_k;
    double *g = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!g) return -1;
    for (int64_t t = 0; t < total_tokens; ++t)
        for (int32_t h = 0; h < num_heads; ++h)
            for (int32_t c = 0; c < d_k; ++c)
                g[(t * num_heads + h) * (int64_t)d_k + c] = g_head ? g_head[t * num_heads + h] : 0.0;
    const int rc = kda_oracle_prefill(num_seqs, total_tokens, num_heads, d_k, d_v, q, k, v, g, beta,
                                      init_state, cu_seqlens, out, final_state, num_threads);
    free(g);
    return rc;
}

/* Gate prologue.  "Understanding Kimi K3's Attention": the log-decay bound
 * equation g_t = g_min Sigmoid(e^{A_h} z_t) (per key channel; A_h the
 * per-head log-scale of the symbol table, z_t the decay logit), and the
 * write strength beta_t = Sigmoid(W_beta x_t) of the symbol table, here from
 * its logit.  Sigmoid(x) = 1 / (1 + e^{-x}); for very negative x, e^{-x}
 * overflows to infinity and the quotient is 0, its limit. */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

int kda_oracle_gate(int32_t total_tokens, int32_t num_heads, int32_t d_k, const double *z,
                    const double *a_log, const double *beta_logit, double *g, double *beta) {
    for (int64_t t = 0; t < total_tokens; ++t)
        for (int32_t h = 0; h < num_heads; ++h) {
            const double scale = exp(a_log[h]);
            for (int32_t c = 0; c < d_k; ++c) {
                const int64_t i = (t * num_heads + h) * (int64_t)d_k + c;
                g[i] = KDA_ORACLE_G_MIN * sigmoid(scale * z[i]);
            }
            beta[t * num_heads + h] = sigmoid(beta_logit[t * num_heads + h]);
        }
    return 0;
}

/* Output gate ("Inside Kimi K3", section "Sequence mixing: fixed-state KDA
 * alongside global MLA": the layer output is W_o [Sigmoid(W_g x_t) .
 * RMSNorm(o~_t)], with o~_t = S_t^T q_t the ungated readout).  The pages do not
 * spell RMSNorm out; it is read here as the root-mean-square normalisation of
 * one head's d_v channels, with an optional per-channel weight and eps inside
 * the square root:
 *
 *   ms      = (1 / d_v) sum_j o~[t,h,j]^2
 *   y[t,h,j] = Sigmoid(gate[t,h,j]) * o~[t,h,j] / sqrt(ms + eps) * w[j]
 *
 * w = 1 when norm_weight is NULL.  eps must be positive (a zero row then gives
 * zeros).  Returns -1 on a bad argument, else 0. */
int kda_oracle_output_gate(int32_t total_tokens, int32_t num_heads, int32_t d_v,
                           const double *o, const double *gate_logit,
                           const double *norm_weight, double eps, double *y) {
    if (total_tokens < 0 || num_heads < 1 || d_v < 1 || !(eps > 0.0) || !o || !gate_logit || !y)
        return -1;
    for (int64_t t = 0; t < total_tokens; ++t)
        for (int32_t h = 0; h < num_heads; ++h) {
            const int64_t row = (t * num_heads + h) * (int64_t)d_v;
            double ss = 0.0;
            for (int32_t j = 0; j < d_v; ++j) ss += o[row + j] * o[row + j];
            const double rinv = 1.0 / sqrt(ss / d_v + eps);
            for (int32_t j = 0; j < d_v; ++j) {
                const double w = norm_weight ? norm_weight[j] : 1.0;
                y[row + j] = sigmoid(gate_logit[row + j]) * o[row + j] * rinv * w;
            }
        }
    return 0;
}

/*
 * The q, k, v prologue ("Understanding Kimi K3's Attention", symbol table:
 * q, k = L2Norm(Swish(ShortConv(W x))), v = Swish(ShortConv(W_v x)); "Inside
 * Kimi K3", section "Sequence mixing": the convolution has width 4; "Hybrid
 * Attention", section "KDA: don't write the same information twice": it is
 * causal).  Read as a per-channel causal convolution over the tokens of one
 * sequence, no bias, followed by Swish(c) = c Sigmoid(c), and for q and k a
 * division by sqrt(sum of squares over the head's channels + eps).
 *
 * Stream s = 0, 1, 2 is q, k, v.  x, y: [3][T][H][d]; conv_weight:
 * [3][H][d][4], tap 3 on the current token, tap 3 - i on the token i places
 * earlier.  conv_state_in / conv_state_out: [N][3][3][H][d], the three
 * inputs before a sequence's first token (entry 0 the oldest) and the last
 * three inputs of the sequence; a NULL state in reads as zeros.
 */
int kda_oracle_qkv_prologue(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                            int32_t d, const int32_t *cu_seqlens, const double *x,
                            const double *conv_weight, const double *conv_state_in, double eps,
                            double *y, double *conv_state_out) {
    if (num_seqs < 0 || total_tokens < 0 || num_heads < 1 || d < 1 || !(eps > 0.0) ||
        !cu_seqlens || !conv_weight || (total_tokens > 0 && (!x || !y)))
        return -1;
    if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != total_tokens) return -1;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    const int64_t H = num_heads, D = d, T = total_tokens;
    for (int32_t n = 0; n < num_seqs; ++n) {
        const int64_t a = cu_seqlens[n], b = cu_seqlens[n + 1];
        for (int s = 0; s < 3; ++s) {
            /* input of stream s at token u of this sequence, head h, channel j */
#define XIN(u, h, j)                                                                        \
    ((u) >= a ? x[((s * T + (u)) * H + (h)) * D + (j)]                                      \
              : (conv_state_in                                                              \
                     ? conv_state_in[((((int64_t)n * 3 + s) * 3 + ((u) - a + 3)) * H + (h)) * D + (j)] \
                     : 0.0))
            for (int64_t t = a; t < b; ++t)
                for (int64_t h = 0; h < H; ++h) {
                    double *row = y + ((s * T + t) * H + h) * D;
                    for (int64_t j = 0; j < D; ++j) {
                        const double *w = conv_weight + ((s * H + h) * D + j) * 4;
                        double c = 0.0;
                        for (int i = 0; i < 4; ++i) c += w[3 - i] * XIN(t - i, h, j);
                        row[j] = c * sigmoid(c);
                    }
                    if (s < 2) {
                        double ss = 0.0;
                        for (int64_t j = 0; j < D; ++j) ss += row[j] * row[j];
                        const double inv = 1.0 / sqrt(ss + eps);
                        for (int64_t j = 0; j < D; ++j) row[j] *= inv;
                    }
                }
            if (conv_state_out)
                for (int p = 0; p < 3; ++p)
                    for (int64_t h = 0; h < H; ++h)
                        for (int64_t j = 0; j < D; ++j)
                            conv_state_out[((((int64_t)n * 3 + s) * 3 + p) * H + h) * D + j] =
                                XIN(b - 3 + p, h, j);
#undef XIN
        }
    }
    return 0;
}

int kda_oracle_decode(int32_t num_seqs, int32_t num_heads, int32_t d_k, int32_t d_v,
                      const double *q, const double *k, const double *v,
                      const double *g, const double *beta, double *state_inout,
                      double *out, int32_t num_threads) {
    /* One token per sequence: the same loop body applied once to each state.
     * The states are read before they are written inside run_one (the copy
     * into the per-thread buffer happens first), so in-place use is safe. */
    return kda_oracle_prefill(num_seqs, num_seqs, num_heads, d_k, d_v, q, k, v, g,
                              beta, state_inout, NULL, out, state_inout, num_threads);
}
