/*
 * kla_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, sequential fp64 CPU statement of Kaczmarz Linear Attention
 * (KLA).  Only the test suite, the smoke check and the benchmark's CPU
 * baseline leg may load this library; the product path never does.  It
 * shares no code, header, table or helper with the CUDA implementation.
 *
 * Source: "Resumo Tecnico: Atencao Linear Kaczmarz (KLA)"
 * (gist.science/pt/paper/2605.08587):
 *   - section "Derivacao Teorica": the write is the state closest to the
 *     decayed previous state S~_{t-1} subject to S^T k_t = v_t;
 *   - section "A Regra de Atualizacao KLA", equation for beta_t:
 *       beta_t = eta_t / (||k_t||_2^2 + eps);
 *   - same section, state update: S_t = S~_{t-1} + beta_t k_t e_t^T with the
 *     residual e_t = v_t - S~_{t-1}^T k_t;
 *   - section "Implementacao": S in R^{dk x dv}, gates (decay and update) of
 *     Gated DeltaNet kept as they are.
 * The decay S~_{t-1} = alpha_t S_{t-1} with a scalar alpha_t per token and
 * head is Gated DeltaNet's gate ("Linear Attention Architectures:
 * Mechanisms, Trade-offs, and Cross-Layer Routing", gist.science
 * 2607.07953, section "Metodologia e Estrutura", item Gated DeltaNet).
 * The read o_t = S_t^T q_t uses the post-update state; it is the read of
 * "Don't Read Everything: A Curvature-Conditioned Query for Linear
 * Attention" (gist.science 2606.01294, section "Integracao", o_t = S_t q)
 * in the dk x dv orientation of the state.
 *
 * Readings where the pages are silent (each also listed in the design
 * notes): the decay uses the current token's alpha_t and is applied before
 * the residual; the write with ||k||^2 + eps == 0 is the limit 0 (beta
 * taken as 0); no normalisation or scaling of q or k is applied.
 *
 * Write-coefficient modes (beta_mode): 0 = Kaczmarz, beta_t as above;
 * 1 = given, beta_t = eta_t itself -- the learned write strength of Gated
 * DeltaNet, which KLA replaces by the Kaczmarz coefficient (KLA summary,
 * "Contribuicoes Principais" item 2 and "Implementacao": only the diagonal
 * B = Diag(beta) of the block solver changes; Linear Attention
 * Architectures, "Metodologia e Estrutura", items DeltaNet and Gated
 * DeltaNet).  alpha == NULL means alpha_t = 1 for every token (no decay:
 * DeltaNet's recurrence).
 *
 * Layouts (dense, row-major, doubles):
 *   q, k : [B, T, H, dk]     v, o : [B, T, H, dv]
 *   alpha, eta : [B, T, H]   S0, S_out : [B, H, dk, dv] (dv fastest)
 * S0 may be NULL (zero initial state).  S_out may be NULL.
 */
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    /* problem */
    int T, H, dk, dv;
    const double *q, *k, *v, *alpha, *eta, *S0;
    double eps;
    int beta_mode;        /* 0: Kaczmarz, 1: given (beta = eta) */
    double *o, *S_out;
    /* varlen: token offsets of each unit's sequence; NULL for fixed length */
    const int *cu_seqlens;
    int n_units;          /* B*H (fixed length) or N*H (varlen) */
    /* work distribution */
    int next_unit;
    pthread_mutex_t lock;
} job_t;

/* One (sequence, head): the per-token recurrence, exactly in the order the
 * update rule states it.  t0 is the first token row of the sequence, len its
 * length; rows of a [*, H, d] tensor for token t and head h sit at
 * ((t0 + t) * H + h) * d. */
static void run_unit(const job_t *J, int unit_seq, int h, long t0, int len,
                     double *S, double *St, double *e)
{
    const int H = J->H, dk = J->dk, dv = J->dv;
    const size_t sd = (size_t)dk * dv;
    const double *S0 = J->S0 ? J->S0 + ((size_t)unit_seq * H + h) * sd : NULL;

    if (S0) memcpy(S, S0, sd * sizeof(double));
    else memset(S, 0, sd * sizeof(double));

    for (int t = 0; t < len; ++t) {
        const size_t row = (size_t)(t0 + t) * H + h;
        const double *kt = J->k + row * dk;
        const double *qt = J->q + row * dk;
        const double *vt = J->v + row * dv;
        const double a = J->alpha ? J->alpha[row] : 1.0;
        const double et = J->eta[row];

        /* Kaczmarz: beta_t = eta_t / (||k_t||^2 + eps); a zero denominator
         * means a zero key with eps = 0, whose write is taken as 0.
         * Given: beta_t = eta_t. */
        double beta = et;
        if (J->beta_mode == 0) {
            double n2 = 0.0;
            for (int i = 0; i < dk; ++i) n2 += kt[i] * kt[i];
            const double den = n2 + J->eps;
            beta = (den == 0.0) ? 0.0 : et / den;
        }

        /* decayed previous state S~ = alpha_t S_{t-1} */
        for (size_t x = 0; x < sd; ++x) St[x] = a * S[x];

        /* residual e_t = v_t - S~^T k_t */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += St[(size_t)i * dv + j] * kt[i];
            e[j] = vt[j] - acc;
        }

        /* S_t = S~ + beta_t k_t e_t^T */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] = St[(size_t)i * dv + j] + beta * kt[i] * e[j];

        /* o_t = S_t^T q_t */
        double *ot = J->o + row * dv;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qt[i];
            ot[j] = acc;
        }
    }

    if (J->S_out)
        memcpy(J->S_out + ((size_t)unit_seq * H + h) * sd, S, sd * sizeof(double));
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const size_t sd = (size_t)J->dk * J->dv;
    double *S = (double *)malloc(sd * sizeof(double));
    double *St = (double *)malloc(sd * sizeof(double));
    double *e = (double *)malloc((size_t)J->dv * sizeof(double));
    if (!S || !St || !e) { free(S); free(St); free(e); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->n_units) break;
        const int seq = u / J->H, h = u % J->H;
        long t0;
        int len;
        if (J->cu_seqlens) {
            t0 = J->cu_seqlens[seq];
            len = J->cu_seqlens[seq + 1] - J->cu_seqlens[seq];
        } else {
            t0 = (long)seq * J->T;
            len = J->T;
        }
        run_unit(J, seq, h, t0, len, S, St, e);
    }
    free(S); free(St); free(e);
    return NULL;
}

static int run_job(job_t *J, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > J->n_units) nthreads = J->n_units > 0 ? J->n_units : 1;
    J->next_unit = 0;
    pthread_mutex_init(&J->lock, NULL);
    int rc = 0;
    if (nthreads == 1) {
        rc = worker(J) != NULL;
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        if (!th) { pthread_mutex_destroy(&J->lock); return 1; }
        int started = 0;
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&th[i], NULL, worker, J) != 0) { rc = 1; break; }
            ++started;
        }
        for (int i = 0; i < started; ++i) {
            void *r = NULL;
            pthread_join(th[i], &r);
            if (r) rc = 1;
        }
        free(th);
    }
    pthread_mutex_destroy(&J->lock);
    return rc;
}

/* Fixed-length batch.  Returns 0 on success, nonzero on bad arguments or
 * allocation failure.  alpha may be NULL (alpha_t = 1). */
int kla_oracle_forward_ex(int B, int T, int H, int dk, int dv,
                          const double *q, const double *k, const double *v,
                          const double *alpha, const double *eta, double eps,
                          const double *S0, double *o, double *S_out, int nthreads,
                          int beta_mode)
{
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 2;
    if (beta_mode != 0 && beta_mode != 1) return 2;
    job_t J;
    memset(&J, 0, sizeof J);
    J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.alpha = alpha; J.eta = eta; J.S0 = S0;
    J.eps = eps; J.o = o; J.S_out = S_out;
    J.beta_mode = beta_mode;
    J.cu_seqlens = NULL;
    J.n_units = B * H;
    return run_job(&J, nthreads);
}

int kla_oracle_forward(int B, int T, int H, int dk, int dv,
                       const double *q, const double *k, const double *v,
                       const double *alpha, const double *eta, double eps,
                       const double *S0, double *o, double *S_out, int nthreads)
{
    return kla_oracle_forward_ex(B, T, H, dk, dv, q, k, v, alpha, eta, eps, S0, o, S_out,
                                 nthreads, 0);
}

/* Packed variable-length batch: sequence n occupies token rows
 * cu_seqlens[n] .. cu_seqlens[n+1]-1 of q, k, v, alpha, eta, o
 * ([total_T, H, *]); S0 and S_out are [N, H, dk, dv]. */
int kla_oracle_forward_varlen_ex(int N, const int *cu_seqlens, int H, int dk, int dv,
                                 const double *q, const double *k, const double *v,
                                 const double *alpha, const double *eta, double eps,
                                 const double *S0, double *o, double *S_out, int nthreads,
                                 int beta_mode)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return 2;
    if (beta_mode != 0 && beta_mode != 1) return 2;
    if (cu_seqlens[0] != 0) return 2;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
    job_t J;
    memset(&J, 0, sizeof J);
    J.T = 0; J.H = H; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.alpha = alpha; J.eta = eta; J.S0 = S0;
    J.eps = eps; J.o = o; J.S_out = S_out;
    J.beta_mode = beta_mode;
    J.cu_seqlens = cu_seqlens;
    J.n_units = N * H;
    return run_job(&J, nthreads);
}

int kla_oracle_forward_varlen(int N, const int *cu_seqlens, int H, int dk, int dv,
                              const double *q, const double *k, const double *v,
                              const double *alpha, const double *eta, double eps,
                              const double *S0, double *o, double *S_out, int nthreads)
{
    return kla_oracle_forward_varlen_ex(N, cu_seqlens, H, dk, dv, q, k, v, alpha, eta, eps, S0,
                                        o, S_out, nthreads, 0);
}
