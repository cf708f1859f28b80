/*
 * ccq_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain sequential fp64 statement of the Curvature-Conditioned Query (CCQ)
 * read-side contraction.  Only the test suite and the benchmark's CPU
 * baseline may load it; it shares no code with the CUDA implementation.
 *
 * Source: "Don't Read Everything: A Curvature-Conditioned Query for Linear
 * Attention" (gist.science 2606.01294):
 *   - section "Derivacao Teorica": Sigma_t = Cov_{<=t}[k], the running
 *     covariance of the keys (the Hessian of the log-partition's Taylor
 *     expansion, C_bar_t - mu_t mu_t^T);
 *   - section "O Mecanismo": q_clean_t = (I - lambda_t Sigma_t) q_t, with a
 *     scalar gate lambda_t per token, and one extra dk x dk matrix and one dk
 *     vector of state per head;
 *   - section "Integracao": the write rule and the state recurrence are
 *     unchanged and the read is o_t = S_t q_clean_t, so the whole CCQ layer
 *     is the unchanged recurrence read with q_clean instead of q.
 * Readings (also in the design notes): Sigma_t is the population covariance
 * (divisor n_t) of every key of the sequence up to and including token t,
 * without decay; lambda_t is an input (the gate's output); the statistics
 * (sum of k k^T, sum of k, count) carry across calls like the state.
 *
 * Layouts (doubles): q, k : [B, T, H, dk]; lambda : [B, T, H];
 * stats: Ms [B, H, dk, dk] (sum of k k^T), ms [B, H, dk] (sum of k),
 * ns [B, H] (count).  Initial statistics may be NULL (zero).
 */
#include <stdlib.h>
#include <string.h>

int ccq_oracle_query(int B, int T, int H, int dk, const double *q, const double *k,
                     const double *lambda, const double *Ms0, const double *ms0,
                     const double *ns0, double *q_clean, double *Ms_out, double *ms_out,
                     double *ns_out)
{
    if (B < 0 || T < 0 || H <= 0 || dk <= 0) return 2;
    double *M = (double *)malloc(sizeof(double) * (size_t)dk * dk);
    double *m = (double *)malloc(sizeof(double) * (size_t)dk);
    double *y = (double *)malloc(sizeof(double) * (size_t)dk);
    if (!M || !m || !y) { free(M); free(m); free(y); return 1; }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const size_t u = (size_t)b * H + h;
            double n = ns0 ? ns0[u] : 0.0;
            if (Ms0) memcpy(M, Ms0 + u * dk * dk, sizeof(double) * (size_t)dk * dk);
            else memset(M, 0, sizeof(double) * (size_t)dk * dk);
            if (ms0) memcpy(m, ms0 + u * dk, sizeof(double) * (size_t)dk);
            else memset(m, 0, sizeof(double) * (size_t)dk);
            for (int t = 0; t < T; ++t) {
                const size_t row = ((size_t)b * T + t) * H + h;
                const double *kt = k + row * dk, *qt = q + row * dk;
                /* statistics up to and including token t */
                n += 1.0;
                for (int i = 0; i < dk; ++i) {
                    m[i] += kt[i];
                    for (int j = 0; j < dk; ++j) M[(size_t)i * dk + j] += kt[i] * kt[j];
                }
                /* Sigma q = (M / n) q - mu (mu . q), mu = m / n */
                double muq = 0.0;
                for (int i = 0; i < dk; ++i) muq += (m[i] / n) * qt[i];
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dk; ++j) acc += (M[(size_t)i * dk + j] / n) * qt[j];
                    y[i] = acc - (m[i] / n) * muq;
                }
                const double lam = lambda[row];
                double *out = q_clean + row * dk;
                for (int i = 0; i < dk; ++i) out[i] = qt[i] - lam * y[i];
            }
            if (Ms_out) memcpy(Ms_out + u * dk * dk, M, sizeof(double) * (size_t)dk * dk);
            if (ms_out) memcpy(ms_out + u * dk, m, sizeof(double) * (size_t)dk);
            if (ns_out) ns_out[u] = n;
        }
    free(M); free(m); free(y);
    return 0;
}
