/*
 * kla_oracle_bwd.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, sequential fp64 gradient of the KLA recurrence (the backward
 * pass of the forward in kla_oracle.c), for the tests of the CUDA backward.
 * Only the test suite may load it; it shares no code with the CUDA library.
 *
 * The forward it differentiates, per (batch, head) and token t ("Resumo
 * Tecnico: Atencao Linear Kaczmarz (KLA)", gist.science 2605.08587, sections
 * "Derivacao Teorica" and "A Regra de Atualizacao KLA"; the decay is Gated
 * DeltaNet's gate, "Linear Attention Architectures", gist.science
 * 2607.07953, "Metodologia e Estrutura"):
 *
 *   n2   = ||k_t||^2,  beta = eta_t / (n2 + eps)   (beta = eta_t when given)
 *   S~   = alpha_t S_{t-1}
 *   e    = v_t - S~^T k_t
 *   S_t  = S~ + beta k_t e^T
 *   o_t  = S_t^T q_t
 *
 * For the scalar L = sum_t <do_t, o_t> + <dS_T, S_T> this file returns
 * dL/dq, dL/dk, dL/dv, dL/dalpha, dL/deta and dL/dS0 by reverse-mode
 * differentiation of those five lines, taken in the opposite order, with
 * the adjoint dS of S_t carried from t = T-1 down to 0:
 *
 *   dS   += q_t do_t^T                     (from o_t = S_t^T q_t)
 *   dq_t  = S_t do_t
 *   dbeta = k_t^T dS e                     (from S_t = S~ + beta k e^T)
 *   dk_t  = beta dS e
 *   de    = beta dS^T k_t
 *   dv_t  = de                              (from e = v - S~^T k)
 *   dS~   = dS - k_t de^T
 *   dk_t += -S~ de
 *   dalpha_t = <dS~, S_{t-1}>               (from S~ = alpha S_{t-1})
 *   dS    = alpha_t dS~                     (the adjoint of S_{t-1})
 *   deta_t = dbeta / (n2 + eps),  dk_t += -2 eta_t dbeta / (n2 + eps)^2 k_t
 *           (Kaczmarz; a zero denominator has beta = 0 and no gradient);
 *   deta_t = dbeta (given).
 *
 * dL/dS0 is the final dS.  The states S_{t-1} are recomputed segment by
 * segment (64 tokens) from checkpoints stored during a first forward sweep.
 *
 * Layouts as kla_oracle.c (doubles, row-major): q, k, dq, dk : [B, T, H, dk];
 * v, do, dv : [B, T, H, dv]; alpha, eta, dalpha, deta : [B, T, H];
 * S0, dS_T, dS0 : [B, H, dk, dv].  alpha NULL = no decay (dalpha then
 * ignored); S0, dS_T NULL = zero; dalpha, dS0 may be NULL.
 */
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define SEG 64

typedef struct {
    int T, H, dk, dv, beta_mode;
    double eps;
    const double *q, *k, *v, *alpha, *eta, *S0, *dout, *dS_T;
    double *dq, *dkey, *dvv, *dalpha, *deta, *dS0;
    int n_units, next_unit;
    pthread_mutex_t lock;
} bjob_t;

typedef struct {
    double *ck;     /* checkpoints: state before token n * SEG */
    double *Sseg;   /* states before each token of one segment */
    double *S, *St, *dS, *dSt, *e, *de;
} bscratch_t;

static double beta_of(const bjob_t *J, const double *kt, double et, double *den_out)
{
    double n2 = 0.0;
    for (int i = 0; i < J->dk; ++i) n2 += kt[i] * kt[i];
    const double den = n2 + J->eps;
    *den_out = den;
    if (J->beta_mode == 1) return et;
    return den == 0.0 ? 0.0 : et / den;
}

/* One forward token: S (S_{t-1} on entry) becomes S_t. */
static void step(const bjob_t *J, size_t row, double *S, double *St, double *e)
{
    const int dk = J->dk, dv = J->dv;
    const double *kt = J->k + row * dk, *vt = J->v + row * dv;
    const double a = J->alpha ? J->alpha[row] : 1.0;
    double den;
    const double beta = beta_of(J, kt, J->eta[row], &den);
    for (size_t x = 0; x < (size_t)dk * dv; ++x) St[x] = a * S[x];
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += St[(size_t)i * dv + j] * kt[i];
        e[j] = vt[j] - acc;
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            S[(size_t)i * dv + j] = St[(size_t)i * dv + j] + beta * kt[i] * e[j];
}

static void bwd_unit(const bjob_t *J, int b, int h, bscratch_t *W)
{
    const int T = J->T, H = J->H, dk = J->dk, dv = J->dv;
    const size_t sd = (size_t)dk * dv;
    const size_t sb = ((size_t)b * H + h) * sd;
    double *S = W->S, *St = W->St, *dS = W->dS, *dSt = W->dSt, *e = W->e, *de = W->de;

    /* forward sweep with a checkpoint at every segment start */
    if (J->S0) memcpy(S, J->S0 + sb, sd * sizeof(double));
    else memset(S, 0, sd * sizeof(double));
    for (int t = 0; t < T; ++t) {
        if (t % SEG == 0) memcpy(W->ck + (size_t)(t / SEG) * sd, S, sd * sizeof(double));
        step(J, (size_t)((long)b * T + t) * H + h, S, St, e);
    }

    if (J->dS_T) memcpy(dS, J->dS_T + sb, sd * sizeof(double));
    else memset(dS, 0, sd * sizeof(double));

    for (int s0 = ((T - 1) / SEG) * SEG; T > 0 && s0 >= 0; s0 -= SEG) {
        const int s1 = s0 + SEG < T ? s0 + SEG : T;
        /* recompute S_{t-1} for t in [s0, s1) */
        memcpy(S, W->ck + (size_t)(s0 / SEG) * sd, sd * sizeof(double));
        for (int t = s0; t < s1; ++t) {
            memcpy(W->Sseg + (size_t)(t - s0) * sd, S, sd * sizeof(double));
            step(J, (size_t)((long)b * T + t) * H + h, S, St, e);
        }
        for (int t = s1 - 1; t >= s0; --t) {
            const size_t row = (size_t)((long)b * T + t) * H + h;
            const double *Sp = W->Sseg + (size_t)(t - s0) * sd;   /* S_{t-1} */
            const double *kt = J->k + row * dk, *qt = J->q + row * dk, *vt = J->v + row * dv;
            const double *dot = J->dout + row * dv;
            const double a = J->alpha ? J->alpha[row] : 1.0;
            const double et = J->eta[row];
            double den;
            const double beta = beta_of(J, kt, et, &den);

            /* recompute S~, e and S_t (S_t into S) */
            for (size_t x = 0; x < sd; ++x) St[x] = a * Sp[x];
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += St[(size_t)i * dv + j] * kt[i];
                e[j] = vt[j] - acc;
            }
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] = St[(size_t)i * dv + j] + beta * kt[i] * e[j];

            /* o_t = S_t^T q_t */
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) dS[(size_t)i * dv + j] += qt[i] * dot[j];
            double *dqt = J->dq + row * dk;
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += S[(size_t)i * dv + j] * dot[j];
                dqt[i] = acc;
            }

            /* S_t = S~ + beta k e^T */
            double dbeta = 0.0;
            double *dkt = J->dkey + row * dk;
            for (int i = 0; i < dk; ++i) {
                double dse = 0.0;
                for (int j = 0; j < dv; ++j) dse += dS[(size_t)i * dv + j] * e[j];
                dbeta += kt[i] * dse;
                dkt[i] = beta * dse;
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += dS[(size_t)i * dv + j] * kt[i];
                de[j] = beta * acc;
            }

            /* e = v - S~^T k */
            double *dvt = J->dvv + row * dv;
            for (int j = 0; j < dv; ++j) dvt[j] = de[j];
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    dSt[(size_t)i * dv + j] = dS[(size_t)i * dv + j] - kt[i] * de[j];
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += St[(size_t)i * dv + j] * de[j];
                dkt[i] -= acc;
            }

            /* S~ = alpha S_{t-1} */
            double da = 0.0;
            for (size_t x = 0; x < sd; ++x) da += dSt[x] * Sp[x];
            if (J->alpha && J->dalpha) J->dalpha[row] = da;
            for (size_t x = 0; x < sd; ++x) dS[x] = a * dSt[x];

            /* beta = eta / (n2 + eps), or beta = eta */
            if (J->beta_mode == 1) {
                J->deta[row] = dbeta;
            } else if (den == 0.0) {
                J->deta[row] = 0.0;
            } else {
                J->deta[row] = dbeta / den;
                const double c = -2.0 * et * dbeta / (den * den);
                for (int i = 0; i < dk; ++i) dkt[i] += c * kt[i];
            }
        }
    }
    if (J->dS0) memcpy(J->dS0 + sb, dS, sd * sizeof(double));
}

static void *bworker(void *arg)
{
    bjob_t *J = (bjob_t *)arg;
    const size_t sd = (size_t)J->dk * J->dv;
    const size_t nseg = (size_t)(J->T + SEG - 1) / SEG + 1;
    bscratch_t W;
    W.ck = (double *)malloc(nseg * sd * sizeof(double));
    W.Sseg = (double *)malloc((size_t)SEG * sd * sizeof(double));
    W.S = (double *)malloc(sd * sizeof(double));
    W.St = (double *)malloc(sd * sizeof(double));
    W.dS = (double *)malloc(sd * sizeof(double));
    W.dSt = (double *)malloc(sd * sizeof(double));
    W.e = (double *)malloc((size_t)J->dv * sizeof(double));
    W.de = (double *)malloc((size_t)J->dv * sizeof(double));
    void *rc = NULL;
    if (!W.ck || !W.Sseg || !W.S || !W.St || !W.dS || !W.dSt || !W.e || !W.de) {
        rc = (void *)1;
    } else {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            const int u = J->next_unit++;
            pthread_mutex_unlock(&J->lock);
            if (u >= J->n_units) break;
            bwd_unit(J, u / J->H, u % J->H, &W);
        }
    }
    free(W.ck); free(W.Sseg); free(W.S); free(W.St); free(W.dS); free(W.dSt);
    free(W.e); free(W.de);
    return rc;
}

/* Fixed-length batch.  Returns 0 on success, nonzero on bad arguments or
 * allocation failure. */
int kla_oracle_backward(int B, int T, int H, int dk, int dv,
                        const double *q, const double *k, const double *v,
                        const double *alpha, const double *eta, double eps,
                        const double *S0, const double *dout, const double *dS_T,
                        double *dq, double *dkey, double *dval, double *dalpha,
                        double *deta, double *dS0, int nthreads, int beta_mode)
{
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 2;
    if (beta_mode != 0 && beta_mode != 1) return 2;
    bjob_t J;
    memset(&J, 0, sizeof J);
    J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.beta_mode = beta_mode; J.eps = eps;
    J.q = q; J.k = k; J.v = v; J.alpha = alpha; J.eta = eta; J.S0 = S0;
    J.dout = dout; J.dS_T = dS_T;
    J.dq = dq; J.dkey = dkey; J.dvv = dval; J.dalpha = dalpha; J.deta = deta; J.dS0 = dS0;
    J.n_units = B * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > J.n_units) nthreads = J.n_units > 0 ? J.n_units : 1;
    pthread_mutex_init(&J.lock, NULL);
    int rc = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) { pthread_mutex_destroy(&J.lock); return 1; }
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, bworker, &J) != 0) { rc = 1; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *r = NULL;
        pthread_join(th[i], &r);
        if (r) rc = 1;
    }
    free(th);
    pthread_mutex_destroy(&J.lock);
    return rc;
}
