/*
 * osdn_oracle.c -- plain fp64 CPU statement of the Online Scaled DeltaNet
 * (OSDN) forward pass, written token by token.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no source, header, table or
 * helper with the CUDA library.
 *
 * Source of every formula: "OSDN: Improving Delta Rule with Provable Online
 * Preconditioning in Linear Attention" (arXiv 2605.13473), as summarised on
 * the gist.science pages (ja/nl/zh/ko), sections 1, 2.1, 2.2 and 2.3:
 *
 *   f_t(S) = 1/2 ||S k_t - v_t||^2                             (section 1)
 *   S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) ktilde_t^T,     (section 2.1)
 *         ktilde_t = d_t (.) k_t
 *   h_t(d) = ((1 - beta_t <d, k_t^2>)^2 - 1) / (2 ||k_t||^2)   (section 2.2)
 *   d_{t+1} = r_t d_t  (-)  eta grad_d h_t(d_t)                (section 2.3)
 *   f_t(S_t) / f_t(S_{t-1}) = (1 - beta_t <d_t, k_t^2>)^2      (section 3,
 *         theorem 5.2: the token-local residual ratio; its geometric mean
 *         over a sequence is the q_geo diagnostic of section 4.2)
 *
 * Readings taken where the pages are silent or garbled:
 *  - the APF step is taken as DESCENT on h (d <- r d - eta grad h); the pages
 *    print "+eta grad h" but call the update online gradient descent on h
 *    (section 2.2), and h is minimised at the gated Newton condition
 *    beta <d,k^2> = 1 (section 3, theorem 5.2);
 *  - no projection or clamp is applied to d_{t+1} (the bar on the left-hand
 *    side of the APF step names no operation);
 *  - ktilde_t uses d_t, the preconditioner before the step of token t;
 *  - grad h := 0 when ||k_t|| = 0 (h is undefined there);
 *  - r = 1 when no retention gate is given (plain OSDN, no APF);
 *  - the optional per-token decay alpha_t (a Gated-DeltaNet-style gate; the
 *    pages name the GDN backbone in section 4 but print no formula) enters as
 *    S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) ktilde_t^T;
 *  - the optional per-channel decay alpha_t in R^K (the Kimi Delta Attention
 *    backbone that section 4 names, with no formula printed: a decay per key
 *    channel in place of GDN's scalar) scales the key columns of the state,
 *    S_t = S_{t-1} Diag(alpha_t) + beta_t (v_t - S_{t-1} Diag(alpha_t) k_t)
 *    ktilde_t^T; with all channels equal it is the scalar gate above;
 *  - the output is o_t = S_t q_t, read from the state after token t, with no
 *    scale on q.
 *
 * Layouts (row-major, all fp64 here):
 *   q, k, ktilde : [B][H][T][K]      v, o : [B][H][T][V]
 *   beta, r, alpha : [B][H][T]       d0, dT : [B][H][K]
 *   alpha_k (per-channel decay) : [B][H][T][K]
 *   S0, ST : [B][H][V][K]  (S[i][j]: i = value row, j = key column)
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* Phase 1: the O(K) scan over the key stream (section 2.2, item 1).      */
/* ---------------------------------------------------------------------- */
static void phase1_sequence(int T, int K, const double *k, const double *beta,
                            const double *r, double eta, const double *d0,
                            double *ktilde, double *dT, double *logratio,
                            double *d /* K scratch */)
{
    double lr = 0.0;
    for (int j = 0; j < K; ++j) d[j] = d0 ? d0[j] : 1.0;
    for (int t = 0; t < T; ++t) {
        const double *kt = k + (size_t)t * K;
        double bt = beta[t];
        double rt = r ? r[t] : 1.0;
        /* ||k_t||^2 and <d_t, k_t^2>: the two quantities the closed form of
         * h_t depends on (section 2.2). */
        double n = 0.0, a = 0.0;
        for (int j = 0; j < K; ++j) {
            double w = kt[j] * kt[j];
            n += w;
            a += d[j] * w;
        }
        /* residual ratio of this token's state write (theorem 5.2):
         * S_t k_t - v_t = (S_{t-1} k_t - v_t)(1 - beta_t <ktilde_t, k_t>) and
         * <ktilde_t, k_t> = <d_t, k_t^2> */
        {
            double y = 1.0 - bt * a;
            lr += log(y * y);
        }
        /* preconditioned key with the preconditioner before this step */
        for (int j = 0; j < K; ++j) ktilde[(size_t)t * K + j] = d[j] * kt[j];
        /* d <- r d - eta * grad_d h_t(d),
         * grad_d h_t(d) = -beta (1 - beta <d,k^2>) k^2 / ||k||^2 */
        for (int j = 0; j < K; ++j) {
            double grad = 0.0;
            if (n > 0.0) grad = -bt * (1.0 - bt * a) * (kt[j] * kt[j]) / n;
            d[j] = rt * d[j] - eta * grad;
        }
    }
    if (dT)
        for (int j = 0; j < K; ++j) dT[j] = d[j];
    if (logratio) *logratio = lr;
}

/* ---------------------------------------------------------------------- */
/* Phase 2: the delta-rule recurrence with ktilde (sections 2.1, 2.2).     */
/* Token by token: the chunkwise form is an implementation choice the      */
/* oracle does not make.                                                   */
/* ---------------------------------------------------------------------- */
static void phase2_sequence(int T, int K, int V, const double *q, const double *k,
                            const double *ktilde, const double *v, const double *beta,
                            const double *alpha, const double *alpha_k, const double *S0,
                            double *o, double *ST, double *S /* V*K scratch */)
{
    for (size_t i = 0; i < (size_t)V * K; ++i) S[i] = S0 ? S0[i] : 0.0;
    for (int t = 0; t < T; ++t) {
        const double *qt = q + (size_t)t * K;
        const double *kt = k + (size_t)t * K;
        const double *kk = ktilde + (size_t)t * K;
        const double *vt = v + (size_t)t * V;
        const double *akt = alpha_k ? alpha_k + (size_t)t * K : NULL;
        double at = alpha ? alpha[t] : 1.0;
        double bt = beta[t];
        for (int i = 0; i < V; ++i) {
            double *Si = S + (size_t)i * K;
            /* decayed state row (per channel, or one scalar), then its
               prediction for k_t */
            double pred = 0.0;
            for (int j = 0; j < K; ++j) {
                Si[j] *= akt ? akt[j] : at;
                pred += Si[j] * kt[j];
            }
            /* u = beta (v - S k): the scaled residual of f_t */
            double u = bt * (vt[i] - pred);
            /* rank-1 write along the preconditioned key */
            double out = 0.0;
            for (int j = 0; j < K; ++j) {
                Si[j] += u * kk[j];
                out += Si[j] * qt[j];
            }
            o[(size_t)t * V + i] = out;
        }
    }
    if (ST) memcpy(ST, S, sizeof(double) * (size_t)V * K);
}

/* ---------------------------------------------------------------------- */
/* Threading over the independent (b,h) sequences.                        */
/* ---------------------------------------------------------------------- */
typedef struct {
    int which; /* 1 = phase 1, 2 = phase 2 */
    int first, last;
    int T, K, V;
    const double *q, *k, *ktilde_in, *v, *beta, *r, *alpha, *alpha_k, *d0, *S0;
    double eta;
    double *ktilde, *dT, *o, *ST, *logratio;
    int failed;
} job_t;

static void *run_job(void *arg)
{
    job_t *jb = (job_t *)arg;
    size_t T = (size_t)jb->T, K = (size_t)jb->K, V = (size_t)jb->V;
    double *scratch = (double *)malloc(sizeof(double) * (jb->which == 1 ? K : V * K));
    if (!scratch) {
        jb->failed = 1;
        return NULL;
    }
    for (int s = jb->first; s < jb->last; ++s) {
        if (jb->which == 1) {
            phase1_sequence(jb->T, jb->K, jb->k + s * T * K, jb->beta + s * T,
                            jb->r ? jb->r + s * T : NULL, jb->eta,
                            jb->d0 ? jb->d0 + s * K : NULL, jb->ktilde + s * T * K,
                            jb->dT ? jb->dT + s * K : NULL,
                            jb->logratio ? jb->logratio + s : NULL, scratch);
        } else {
            phase2_sequence(jb->T, jb->K, jb->V, jb->q + s * T * K, jb->k + s * T * K,
                            jb->ktilde_in + s * T * K, jb->v + s * T * V, jb->beta + s * T,
                            jb->alpha ? jb->alpha + s * T : NULL,
                            jb->alpha_k ? jb->alpha_k + s * T * K : NULL,
                            jb->S0 ? jb->S0 + s * V * K : NULL, jb->o + s * T * V,
                            jb->ST ? jb->ST + s * V * K : NULL, scratch);
        }
    }
    free(scratch);
    return NULL;
}

static int run_threads(job_t *proto, int nseq, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nseq) nthreads = nseq;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    if (!th || !jobs) {
        free(th);
        free(jobs);
        return -1;
    }
    int rc = 0;
    char *joined = (char *)calloc((size_t)nthreads, 1);
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = *proto;
        jobs[i].first = (int)((long long)nseq * i / nthreads);
        jobs[i].last = (int)((long long)nseq * (i + 1) / nthreads);
        if (pthread_create(&th[i], NULL, run_job, &jobs[i]) == 0) {
            if (joined) joined[i] = 1;
            else pthread_join(th[i], NULL);
        } else {
            run_job(&jobs[i]); /* run inline if no thread could be made */
        }
    }
    for (int i = 0; i < nthreads; ++i) {
        if (joined && joined[i]) pthread_join(th[i], NULL);
        if (jobs[i].failed) rc = -1;
    }
    free(joined);
    free(th);
    free(jobs);
    return rc;
}

/* Phase 1 over B*H sequences.  r, d0, dT, logratio may be NULL (r = 1,
 * d0 = 1).  logratio[b*H + h] = sum_t log((1 - beta_t <d_t, k_t^2>)^2), the
 * log of the product of the sequence's token residual ratios. */
int oracle_precond_scan(int B, int H, int T, int K, const double *k, const double *beta,
                        const double *r, double eta, const double *d0, double *ktilde,
                        double *dT, double *logratio, int nthreads)
{
    if (B < 1 || H < 1 || T < 0 || K < 1 || !k || !beta || !ktilde) return -1;
    if (T == 0) {
        for (size_t i = 0; dT && i < (size_t)B * H * K; ++i) dT[i] = d0 ? d0[i] : 1.0;
        for (size_t i = 0; logratio && i < (size_t)B * H; ++i) logratio[i] = 0.0;
        return 0;
    }
    job_t p;
    memset(&p, 0, sizeof(p));
    p.which = 1;
    p.T = T;
    p.K = K;
    p.k = k;
    p.beta = beta;
    p.r = r;
    p.eta = eta;
    p.d0 = d0;
    p.ktilde = ktilde;
    p.dT = dT;
    p.logratio = logratio;
    return run_threads(&p, B * H, nthreads);
}

/* Phase 2 over B*H sequences.  alpha, S0, ST may be NULL (alpha = 1, S0 = 0). */
int oracle_delta_fwd(int B, int H, int T, int K, int V, const double *q, const double *k,
                     const double *ktilde, const double *v, const double *beta,
                     const double *alpha, const double *S0, double *o, double *ST,
                     int nthreads)
{
    if (B < 1 || H < 1 || T < 0 || K < 1 || V < 1) return -1;
    if (T > 0 && (!q || !k || !ktilde || !v || !beta || !o)) return -1;
    if (T == 0) {
        for (size_t i = 0; ST && i < (size_t)B * H * V * K; ++i) ST[i] = S0 ? S0[i] : 0.0;
        return 0;
    }
    job_t p;
    memset(&p, 0, sizeof(p));
    p.which = 2;
    p.T = T;
    p.K = K;
    p.V = V;
    p.q = q;
    p.k = k;
    p.ktilde_in = ktilde;
    p.v = v;
    p.beta = beta;
    p.alpha = alpha;
    p.S0 = S0;
    p.o = o;
    p.ST = ST;
    return run_threads(&p, B * H, nthreads);
}

/* Phase 2 with a per-channel decay alpha_k [B][H][T][K] (NULL: no decay)
 * over B*H sequences.  S0, ST may be NULL. */
int oracle_delta_fwd_kda(int B, int H, int T, int K, int V, const double *q, const double *k,
                         const double *ktilde, const double *v, const double *beta,
                         const double *alpha_k, const double *S0, double *o, double *ST,
                         int nthreads)
{
    if (B < 1 || H < 1 || T < 0 || K < 1 || V < 1) return -1;
    if (T > 0 && (!q || !k || !ktilde || !v || !beta || !o)) return -1;
    if (T == 0) {
        for (size_t i = 0; ST && i < (size_t)B * H * V * K; ++i) ST[i] = S0 ? S0[i] : 0.0;
        return 0;
    }
    job_t p;
    memset(&p, 0, sizeof(p));
    p.which = 2;
    p.T = T;
    p.K = K;
    p.V = V;
    p.q = q;
    p.k = k;
    p.ktilde_in = ktilde;
    p.v = v;
    p.beta = beta;
    p.alpha_k = alpha_k;
    p.S0 = S0;
    p.o = o;
    p.ST = ST;
    return run_threads(&p, B * H, nthreads);
}
