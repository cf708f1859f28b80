// Backward pass of the chunkwise KLA forward on CUDA cores, fp32 arithmetic.
//
// The forward is the blockwise solver of the Kaczmarz Linear Attention
// summary (gist.science 2605.08587, sections "Implementacao" and "A Regra de
// Atualizacao KLA"): for one chunk of C = 64 tokens starting from state S,
//
//   g = cumsum(log alpha), Gamma_ts = exp(g_t - g_s) (s <= t)
//   beta = eta / (||k||^2 + eps)            (beta = eta in the given mode)
//   T    = (I + strict_lower(diag(beta) Gamma o K K^T))^{-1}
//   R    = diag(beta) (V - diag(exp g) K S),   U = T R
//   O    = diag(exp g) Q S + lower(Gamma o Q K^T) U
//   S'   = exp(g_C) S + (diag(exp(g_C - g)) K)^T U
//
// and its reverse-mode derivative, given dO and dS' (the gradient of the
// state at the chunk's end), is
//
//   dU  = A_qk^T dO + diag(exp(g_C - g)) K dS'
//   dR  = T^T dU
//   dS  = exp(g_C) dS' + Q^T diag(exp g) dO - K^T diag(beta exp g) dR
//   dV  = diag(beta) dR
//   dA_qk = lower(dO U^T),   dA_kk = -strict_lower(dR U^T)
//   dQ  = diag(exp g) dO S^T + (dA_qk o Gamma) K
//   dK  = (dA_qk o Gamma)^T Q + X K + X^T K - diag(beta exp g) dR S^T
//         + diag(exp(g_C - g)) U dS'^T,     X = diag(beta) (dA_kk o Gamma)
//   dbeta_t = (V - diag(exp g) K S)_t . dR_t + sum_s (dA_kk o Gamma)_ts (k_t . k_s)
//   dg_t  from every exp(g) factor above; dlog(alpha) = reverse cumsum of dg
//   deta = dbeta / (||k||^2 + eps),  dK += -2 eta dbeta / (||k||^2 + eps)^2 k
//
// Three launches:
//   1. the chunkwise forward on the CUDA cores, recording S at every chunk
//      start (no outputs);
//   2. bwd_dstate_kernel: per (batch, head, 32 columns of dv) the chunks in
//      reverse, carrying dS through the dS line above and recording dS' of
//      every chunk (the columns of dS evolve independently);
//   3. bwd_grads_kernel: per (chunk, batch, head), in parallel, every token
//      gradient from the recorded S and dS'.

#include <cuda_bf16.h>

#include "kla_internal.h"

namespace kla {
namespace {

constexpr int C = kChunk;
constexpr int NT = 256;
constexpr int DVB = 32;   // dv columns per CTA of the state-gradient chain

__device__ __forceinline__ float ld_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_out(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// Per-chunk vectors.  Tail positions of a partial chunk are identity tokens
// (k = q = v = 0, alpha = 1, eta = 0, beta = 0).
struct Vec {
    float alpha[C], eta[C], g[C], beta[C], eg[C], egc[C], den[C];
};

template <typename Tin, int D>
__device__ void load_kq(float (*K)[D + 1], float (*Q)[D + 1], Vec &v, const BwdProblem &p,
                        long row0, int nc, int h, int tid) {
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *q = static_cast<const Tin *>(p.q);
    for (int x = tid; x < C * D; x += NT) {
        const int t = x / D, i = x % D;
        float kv = 0.f, qv = 0.f;
        if (t < nc) {
            const size_t r = (size_t)(row0 + t) * p.H + h;
            kv = ld_in(k, r * D + i);
            qv = ld_in(q, r * D + i);
        }
        K[t][i] = kv;
        Q[t][i] = qv;
    }
    if (tid < C) {
        const bool ok = tid < nc;
        const size_t r = (size_t)(row0 + tid) * p.H + h;
        v.alpha[tid] = (ok && p.alpha) ? p.alpha[r] : 1.f;
        v.eta[tid] = ok ? p.eta[r] : 0.f;
    }
}

// beta, ||k||^2 + eps and the in-chunk log-decay prefix sums (after K, alpha
// and eta are in shared memory).
template <int D>
__device__ void chunk_vectors(const float (*K)[D + 1], Vec &v, float eps, int beta_mode, int nc,
                              int tid) {
    if (tid < C) {
        float n2 = 0.f;
        for (int i = 0; i < D; ++i) n2 = fmaf(K[tid][i], K[tid][i], n2);
        const float den = n2 + eps;
        v.den[tid] = den;
        const float b = beta_mode ? v.eta[tid] : (den != 0.f ? v.eta[tid] / den : 0.f);
        v.beta[tid] = tid < nc ? b : 0.f;
    } else if (tid < C + 32) {
        const int lane = tid - C;
        double a0 = (double)logf(v.alpha[lane]);
        double a1 = (double)logf(v.alpha[lane + 32]);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double u0 = __shfl_up_sync(0xffffffffu, a0, off);
            const double u1 = __shfl_up_sync(0xffffffffu, a1, off);
            if (lane >= off) { a0 += u0; a1 += u1; }
        }
        a1 += __shfl_sync(0xffffffffu, a0, 31);
        const double gC = __shfl_sync(0xffffffffu, a1, 31);
        v.g[lane] = (float)a0;
        v.g[lane + 32] = (float)a1;
        v.eg[lane] = (float)exp(a0);
        v.eg[lane + 32] = (float)exp(a1);
        v.egc[lane] = (float)exp(gC - a0);
        v.egc[lane + 32] = (float)exp(gC - a1);
    }
}

__device__ __forceinline__ float gam(const Vec &v, int t, int s) { return expf(v.g[t] - v.g[s]); }

// Gram products over the chunk, 4 x 4 register blocks on the lower triangle.
// kApply: Mkk = strict_lower(beta Gamma o K K^T), Mqk = lower(Gamma o Q K^T);
// otherwise the raw products (strict lower K K^T, lower Q K^T); zero above.
template <int D, bool kApply>
__device__ void gram(const float (*K)[D + 1], const float (*Q)[D + 1], const Vec &v,
                     float (*Mkk)[C + 1], float (*Mqk)[C + 1], int tid) {
    const int bt = tid / 16, bs = tid % 16;
    float akk[4][4], aqk[4][4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) akk[m][n] = aqk[m][n] = 0.f;
    if (bs <= bt) {
        for (int i = 0; i < D; ++i) {
            float kt[4], qt[4], ks[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                kt[m] = K[bt * 4 + m][i];
                qt[m] = Q[bt * 4 + m][i];
                ks[m] = K[bs * 4 + m][i];
            }
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    akk[m][n] = fmaf(kt[m], ks[n], akk[m][n]);
                    aqk[m][n] = fmaf(qt[m], ks[n], aqk[m][n]);
                }
        }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int t = bt * 4 + m, s = bs * 4 + n;
            const float ga = kApply ? ((s <= t) ? gam(v, t, s) : 0.f) : 1.f;
            const float bk = kApply ? v.beta[t] : 1.f;
            Mkk[t][s] = (s < t) ? bk * ga * akk[m][n] : 0.f;
            Mqk[t][s] = (s <= t) ? ga * aqk[m][n] : 0.f;
        }
}

// T = (I + A_kk)^{-1} by forward substitution, one column per thread (tid < C).
// kRaw: A_kk(t, s) = beta_t Gamma_ts G(t, s) from the raw strict-lower G.
template <bool kRaw>
__device__ void solve_t(const float (*A)[C + 1], const Vec &v, float (*Tm)[C + 1], int tid) {
    if (tid >= C) return;
    const int j = tid;
    for (int t = 0; t < C; ++t) {
        float x = (t == j) ? 1.f : 0.f;
        for (int s = j; s < t; ++s) {
            const float a = kRaw ? v.beta[t] * gam(v, t, s) * A[t][s] : A[t][s];
            x = fmaf(-a, Tm[s][j], x);
        }
        Tm[t][j] = x;
    }
}

// ---------------------------------------------------------------- dS chain
template <int D>
struct DsSmem {
    float K[C][D + 1], Q[C][D + 1];
    float Akk[C][C + 1], Aqk[C][C + 1], Tm[C][C + 1];
    float dS[D][DVB + 1];
    float dO[C][DVB + 1], dU[C][DVB + 1], dR[C][DVB + 1];
    Vec v;
};

template <typename Tin, int D>
__global__ void __launch_bounds__(NT, 1) bwd_dstate_kernel(BwdProblem p, int nch, float *dS_chk) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    DsSmem<D> &sm = *reinterpret_cast<DsSmem<D> *>(smem_raw);
    const int tid = threadIdx.x;
    const int unit = blockIdx.x, b = unit / p.H, h = unit % p.H;
    const int jb = blockIdx.y * DVB;
    if (p.status != nullptr && *(volatile unsigned *)p.status != kDevOk) return;
    const Tin *dout = static_cast<const Tin *>(p.dout);
    const size_t sbase = (size_t)unit * D * D;

    for (int x = tid; x < D * DVB; x += NT) {
        const int i = x / DVB, j = x % DVB;
        sm.dS[i][j] = p.dS_T ? p.dS_T[sbase + (size_t)i * D + jb + j] : 0.f;
    }
    for (int c = nch - 1; c >= 0; --c) {
        const long row0 = (long)b * p.T + (long)c * C;
        const int nc = min(C, p.T - c * C);
        __syncthreads();   // the previous chunk is done with every tile
        float *rec = dS_chk + ((size_t)unit * nch + c) * D * D;   // dS' of chunk c
        for (int x = tid; x < D * DVB; x += NT) {
            const int i = x / DVB, j = x % DVB;
            rec[(size_t)i * D + jb + j] = sm.dS[i][j];
        }
        load_kq<Tin, D>(sm.K, sm.Q, sm.v, p, row0, nc, h, tid);
        for (int x = tid; x < C * DVB; x += NT) {
            const int t = x / DVB, j = x % DVB;
            sm.dO[t][j] = t < nc ? ld_in(dout, ((size_t)(row0 + t) * p.H + h) * D + jb + j) : 0.f;
        }
        __syncthreads();
        chunk_vectors<D>(sm.K, sm.v, p.eps, p.beta_mode, nc, tid);
        __syncthreads();
        gram<D, true>(sm.K, sm.Q, sm.v, sm.Akk, sm.Aqk, tid);
        __syncthreads();
        {   // dU = A_qk^T dO + diag(exp(g_C - g)) K dS'
            const int t = tid / 4, jq = (tid % 4) * 8;
            float acc[8];
#pragma unroll
            for (int n = 0; n < 8; ++n) acc[n] = 0.f;
            for (int s = t; s < C; ++s) {
                const float a = sm.Aqk[s][t];
#pragma unroll
                for (int n = 0; n < 8; ++n) acc[n] = fmaf(a, sm.dO[s][jq + n], acc[n]);
            }
            const float e = sm.v.egc[t];
            for (int i = 0; i < D; ++i) {
                const float kw = e * sm.K[t][i];
#pragma unroll
                for (int n = 0; n < 8; ++n) acc[n] = fmaf(kw, sm.dS[i][jq + n], acc[n]);
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) sm.dU[t][jq + n] = acc[n];
        }
        solve_t<false>(sm.Akk, sm.v, sm.Tm, tid);
        __syncthreads();
        {   // dR = T^T dU
            const int t = tid / 4, jq = (tid % 4) * 8;
            float acc[8];
#pragma unroll
            for (int n = 0; n < 8; ++n) acc[n] = 0.f;
            for (int s = t; s < C; ++s) {
                const float a = sm.Tm[s][t];
#pragma unroll
                for (int n = 0; n < 8; ++n) acc[n] = fmaf(a, sm.dU[s][jq + n], acc[n]);
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) sm.dR[t][jq + n] = acc[n];
        }
        __syncthreads();
        {   // dS <- exp(g_C) dS' + Q^T diag(exp g) dO - K^T diag(beta exp g) dR
            constexpr int TPR = NT / D;
            constexpr int JPT = DVB / TPR;
            const int i = tid / TPR, j0 = (tid % TPR) * JPT;
            const float egC = sm.v.eg[C - 1];
            float acc[JPT];
#pragma unroll
            for (int n = 0; n < JPT; ++n) acc[n] = egC * sm.dS[i][j0 + n];
            for (int t = 0; t < nc; ++t) {
                const float wq = sm.Q[t][i] * sm.v.eg[t];
                const float wk = -sm.K[t][i] * sm.v.beta[t] * sm.v.eg[t];
#pragma unroll
                for (int n = 0; n < JPT; ++n)
                    acc[n] = fmaf(wq, sm.dO[t][j0 + n], fmaf(wk, sm.dR[t][j0 + n], acc[n]));
            }
#pragma unroll
            for (int n = 0; n < JPT; ++n) sm.dS[i][j0 + n] = acc[n];
        }
    }
    __syncthreads();
    if (p.dS0) {
        for (int x = tid; x < D * DVB; x += NT) {
            const int i = x / DVB, j = x % DVB;
            p.dS0[sbase + (size_t)i * D + jb + j] = sm.dS[i][j];
        }
    }
}

// ------------------------------------------------------------ token gradients
template <int D>
struct GrSmem {
    float K[C][D + 1], Q[C][D + 1];
    float M0[C][C + 1];   // raw strict-lower K K^T
    float M1[C][C + 1];   // raw lower Q K^T
    float M2[C][C + 1];   // T, then dA_qk, then dA_qk o Gamma
    float tA[C][D + 1];   // U
    float tB[C][D + 1];   // V - diag(exp g) K S, then dR
    float tC[C][D + 1];   // dO, then dU, then dA_kk and X (as [C][C + 1])
    Vec v;
    float dbeta[C], dg[C], dgcol[C], red[NT / 32];
};

template <typename Tin, int D>
__global__ void __launch_bounds__(NT, 1) bwd_grads_kernel(BwdProblem p, int nch,
                                                          const float *S_chk,
                                                          const float *dS_chk) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    GrSmem<D> &sm = *reinterpret_cast<GrSmem<D> *>(smem_raw);
    float(*dAkk)[C + 1] = reinterpret_cast<float(*)[C + 1]>(&sm.tC[0][0]);
    constexpr int CPT = D / 4;   // columns per thread: cq + 4 x
    const int tid = threadIdx.x;
    const int c = blockIdx.x, unit = blockIdx.y, b = unit / p.H, h = unit % p.H;
    if (p.status != nullptr && *(volatile unsigned *)p.status != kDevOk) return;
    const long row0 = (long)b * p.T + (long)c * C;
    const int nc = min(C, p.T - c * C);
    const float *S = S_chk + ((size_t)unit * nch + c) * D * D;     // state at the chunk start
    const float *dSp = dS_chk + ((size_t)unit * nch + c) * D * D;  // gradient at its end
    const Tin *dout = static_cast<const Tin *>(p.dout);
    const Tin *vin = static_cast<const Tin *>(p.v);
    const int t = tid >> 2, cq = tid & 3;
    const size_t rt = (size_t)(row0 + t) * p.H + h;   // token row of this thread's t
    const bool live = t < nc;

    load_kq<Tin, D>(sm.K, sm.Q, sm.v, p, row0, nc, h, tid);
    for (int x = tid; x < C * D; x += NT) {
        const int tt = x / D, j = x % D;
        sm.tC[tt][j] = tt < nc ? ld_in(dout, ((size_t)(row0 + tt) * p.H + h) * D + j) : 0.f;
    }
    __syncthreads();
    chunk_vectors<D>(sm.K, sm.v, p.eps, p.beta_mode, nc, tid);
    __syncthreads();
    gram<D, false>(sm.K, sm.Q, sm.v, sm.M0, sm.M1, tid);
    {   // V - diag(exp g) K S
        float acc[CPT];
#pragma unroll
        for (int x = 0; x < CPT; ++x) acc[x] = 0.f;
        for (int i = 0; i < D; ++i) {
            const float kti = sm.K[t][i];
            const float *Si = S + (size_t)i * D + cq;
#pragma unroll
            for (int x = 0; x < CPT; ++x) acc[x] = fmaf(kti, Si[4 * x], acc[x]);
        }
        const float e = sm.v.eg[t];
#pragma unroll
        for (int x = 0; x < CPT; ++x) {
            const float vv = live ? ld_in(vin, rt * D + cq + 4 * x) : 0.f;
            sm.tB[t][cq + 4 * x] = vv - e * acc[x];
        }
    }
    __syncthreads();
    solve_t<true>(sm.M0, sm.v, sm.M2, tid);
    __syncthreads();
    {   // U = T diag(beta) (V - e^g K S);  dU = A_qk^T dO + diag(exp(g_C - g)) K dS'
        float u[CPT], du[CPT];
#pragma unroll
        for (int x = 0; x < CPT; ++x) u[x] = du[x] = 0.f;
        for (int s = 0; s <= t; ++s) {
            const float a = sm.M2[t][s] * sm.v.beta[s];
#pragma unroll
            for (int x = 0; x < CPT; ++x) u[x] = fmaf(a, sm.tB[s][cq + 4 * x], u[x]);
        }
        for (int s = t; s < C; ++s) {
            const float a = gam(sm.v, s, t) * sm.M1[s][t];
#pragma unroll
            for (int x = 0; x < CPT; ++x) du[x] = fmaf(a, sm.tC[s][cq + 4 * x], du[x]);
        }
        const float e = sm.v.egc[t];
        for (int i = 0; i < D; ++i) {
            const float kw = e * sm.K[t][i];
            const float *Di = dSp + (size_t)i * D + cq;
#pragma unroll
            for (int x = 0; x < CPT; ++x) du[x] = fmaf(kw, Di[4 * x], du[x]);
        }
        __syncthreads();   // dO in tC fully read
#pragma unroll
        for (int x = 0; x < CPT; ++x) {
            sm.tA[t][cq + 4 * x] = u[x];
            sm.tC[t][cq + 4 * x] = du[x];
        }
    }
    __syncthreads();
    {   // dR = T^T dU; dV; dbeta and dg from R = diag(beta)(V - e^g K S)
        float dr[CPT];
#pragma unroll
        for (int x = 0; x < CPT; ++x) dr[x] = 0.f;
        for (int s = t; s < C; ++s) {
            const float a = sm.M2[s][t];
#pragma unroll
            for (int x = 0; x < CPT; ++x) dr[x] = fmaf(a, sm.tC[s][cq + 4 * x], dr[x]);
        }
        float p1 = 0.f, p2 = 0.f;
        Tin *dvo = static_cast<Tin *>(p.dv);
        const float bt = sm.v.beta[t];
#pragma unroll
        for (int x = 0; x < CPT; ++x) {
            const float vv = live ? ld_in(vin, rt * D + cq + 4 * x) : 0.f;
            p1 = fmaf(sm.tB[t][cq + 4 * x], dr[x], p1);
            p2 = fmaf(vv, dr[x], p2);
            if (live) st_out(dvo, rt * D + cq + 4 * x, bt * dr[x]);
        }
        p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
        p2 += __shfl_xor_sync(0xffffffffu, p2, 1);
        p2 += __shfl_xor_sync(0xffffffffu, p2, 2);
        if (cq == 0) {
            sm.dbeta[t] = p1;
            sm.dg[t] = bt * (p1 - p2);   // -beta e^g (K S)_t . dR_t
        }
        __syncthreads();   // V - e^g K S, dU and T fully read
#pragma unroll
        for (int x = 0; x < CPT; ++x) sm.tB[t][cq + 4 * x] = dr[x];
    }
    __syncthreads();
    {   // dA_qk = lower(dO U^T) -> M2;  dA_kk = -strict_lower(dR U^T) -> tC
        constexpr int SPT = C / 4;
        float da[SPT], dk2[SPT];
#pragma unroll
        for (int x = 0; x < SPT; ++x) da[x] = dk2[x] = 0.f;
        for (int j = 0; j < D; ++j) {
            const float o = live ? ld_in(dout, rt * D + j) : 0.f;
            const float r = sm.tB[t][j];
#pragma unroll
            for (int x = 0; x < SPT; ++x) {
                const float us = sm.tA[cq + 4 * x][j];
                da[x] = fmaf(o, us, da[x]);
                dk2[x] = fmaf(r, us, dk2[x]);
            }
        }
#pragma unroll
        for (int x = 0; x < SPT; ++x) {
            const int s = cq + 4 * x;
            sm.M2[t][s] = s <= t ? da[x] : 0.f;
            dAkk[t][s] = s < t ? -dk2[x] : 0.f;
        }
    }
    __syncthreads();
    // dg, dbeta from the Gamma and beta factors of A_qk and A_kk: row sums
    // (threads 0..63) and column sums (threads 64..127)
    if (tid < C) {
        const int r = tid;
        float sg = 0.f, sb = 0.f;
        for (int s = 0; s <= r; ++s) {
            const float ga = gam(sm.v, r, s);
            sg = fmaf(sm.M2[r][s], ga * sm.M1[r][s], sg);
            if (s < r) {
                const float x = dAkk[r][s] * ga * sm.M0[r][s];
                sb += x;
                sg = fmaf(sm.v.beta[r], x, sg);
            }
        }
        sm.dg[r] += sg;
        sm.dbeta[r] += sb;
    } else if (tid < 2 * C) {
        const int s = tid - C;
        float sg = 0.f;
        for (int r = s; r < C; ++r) {
            const float ga = gam(sm.v, r, s);
            sg = fmaf(sm.M2[r][s], ga * sm.M1[r][s], sg);
            if (s < r) sg = fmaf(sm.v.beta[r], dAkk[r][s] * ga * sm.M0[r][s], sg);
        }
        sm.dgcol[s] = sg;
    }
    __syncthreads();
    {   // M2 <- dA_qk o Gamma;  tC <- X = diag(beta) (dA_kk o Gamma)
        constexpr int SPT = C / 4;
#pragma unroll
        for (int x = 0; x < SPT; ++x) {
            const int s = cq + 4 * x;
            const float ga = s <= t ? gam(sm.v, t, s) : 0.f;
            sm.M2[t][s] *= ga;
            dAkk[t][s] *= sm.v.beta[t] * ga;
        }
        if (tid < C) sm.dg[tid] -= sm.dgcol[tid];
    }
    __syncthreads();
    {   // dQ and dK of token t, dims i = cq + 4 x
        float dq[CPT], dkk[CPT], pq[CPT], pr[CPT], pu[CPT];
#pragma unroll
        for (int x = 0; x < CPT; ++x) dq[x] = dkk[x] = pq[x] = pr[x] = pu[x] = 0.f;
        // dO S^T, dR S^T and U dS'^T for rows i of S and dS'
        for (int j = 0; j < D; ++j) {
            const float o = live ? ld_in(dout, rt * D + j) : 0.f;
            const float r = sm.tB[t][j], u = sm.tA[t][j];
#pragma unroll
            for (int x = 0; x < CPT; ++x) {
                const size_t ij = (size_t)(cq + 4 * x) * D + j;
                const float sv = S[ij];
                pq[x] = fmaf(o, sv, pq[x]);
                pr[x] = fmaf(r, sv, pr[x]);
                pu[x] = fmaf(u, dSp[ij], pu[x]);
            }
        }
        // (dA_qk o Gamma) K, its transpose times Q, X K and X^T K
        for (int s = 0; s < C; ++s) {
            const float a_ts = sm.M2[t][s], a_st = sm.M2[s][t];
            const float x_ts = dAkk[t][s], x_st = dAkk[s][t];
#pragma unroll
            for (int x = 0; x < CPT; ++x) {
                const int i = cq + 4 * x;
                dq[x] = fmaf(a_ts, sm.K[s][i], dq[x]);
                dkk[x] = fmaf(a_st, sm.Q[s][i], dkk[x]);
                dkk[x] = fmaf(x_ts + x_st, sm.K[s][i], dkk[x]);
            }
        }
        const float eg = sm.v.eg[t], egc = sm.v.egc[t], bt = sm.v.beta[t];
        float gq = 0.f, gk = 0.f;
#pragma unroll
        for (int x = 0; x < CPT; ++x) {
            const int i = cq + 4 * x;
            dq[x] = fmaf(eg, pq[x], dq[x]);
            dkk[x] = fmaf(-bt * eg, pr[x], dkk[x]);
            dkk[x] = fmaf(egc, pu[x], dkk[x]);
            gq = fmaf(sm.Q[t][i], pq[x], gq);
            gk = fmaf(sm.K[t][i], pu[x], gk);
        }
        gq += __shfl_xor_sync(0xffffffffu, gq, 1);
        gq += __shfl_xor_sync(0xffffffffu, gq, 2);
        gk += __shfl_xor_sync(0xffffffffu, gk, 1);
        gk += __shfl_xor_sync(0xffffffffu, gk, 2);
        // the gradient through beta's key norm
        const float db = sm.dbeta[t];
        float cn = 0.f;
        if (p.beta_mode == 0 && sm.v.den[t] != 0.f) {
            const float den = sm.v.den[t];
            cn = -2.f * sm.v.eta[t] * db / (den * den);
        }
        if (live) {
            Tin *dqo = static_cast<Tin *>(p.dq);
            Tin *dko = static_cast<Tin *>(p.dk);
#pragma unroll
            for (int x = 0; x < CPT; ++x) {
                const int i = cq + 4 * x;
                st_out(dqo, rt * D + i, dq[x]);
                st_out(dko, rt * D + i, fmaf(cn, sm.K[t][i], dkk[x]));
            }
        }
        // dg: exp(g) of the Q S read, exp(g_C - g) of the state write
        const float wk = egc * gk;
        if (cq == 0) sm.dg[t] += eg * gq - wk;
        // dg_C: the state write and exp(g_C) S
        float red = (cq == 0) ? wk : 0.f;
        for (int x = tid; x < D * D; x += NT) red = fmaf(sm.v.eg[C - 1] * dSp[x], S[x], red);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) red += __shfl_xor_sync(0xffffffffu, red, off);
        if ((tid & 31) == 0) sm.red[tid >> 5] = red;
    }
    __syncthreads();
    if (tid < 32) {   // dg_C onto g_{C-1}; reverse cumulative sum -> dlog(alpha)
        float gc = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) gc += sm.red[w];
        const int lane = tid;
        float d0 = sm.dg[lane], d1 = sm.dg[lane + 32];
        if (lane == 31) d1 += gc;
        // reverse inclusive scan over 64 positions: suffix sums
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float u0 = __shfl_down_sync(0xffffffffu, d0, off);
            const float u1 = __shfl_down_sync(0xffffffffu, d1, off);
            if (lane + off < 32) { d0 += u0; d1 += u1; }
        }
        d0 += __shfl_sync(0xffffffffu, d1, 0);
        const float dl[2] = {d0, d1};
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
            const int tt = lane + 32 * q2;
            if (tt < nc) {
                const size_t r = (size_t)(row0 + tt) * p.H + h;
                if (p.dalpha && p.alpha) p.dalpha[r] = dl[q2] / sm.v.alpha[tt];
                if (p.deta) {
                    const float db = sm.dbeta[tt];
                    const float den = sm.v.den[tt];
                    p.deta[r] = p.beta_mode ? db : (den != 0.f ? db / den : 0.f);
                }
            }
        }
    }
}

template <typename Tin, int D>
cudaError_t launch_bwd_t(const BwdProblem &p, cudaStream_t s) {
    const int nch = (p.T + C - 1) / C;
    const int units = p.B * p.H;
    float *S_chk = static_cast<float *>(p.ws);
    float *dS_chk = S_chk + (size_t)units * nch * D * D;
    // 1. states at the chunk starts (the forward, no outputs)
    Problem f{};
    f.q = p.q; f.k = p.k; f.v = p.v; f.alpha = p.alpha; f.eta = p.eta; f.eps = p.eps;
    f.S0 = p.S0; f.o = nullptr; f.S_T = nullptr; f.cu_seqlens = nullptr;
    f.n_seq = p.B; f.T = p.T; f.total_T = p.B * p.T; f.H = p.H; f.d = D; f.dtype = p.dtype;
    f.beta_mode = p.beta_mode; f.S_chk = S_chk; f.status = p.status;
    cudaError_t e = launch_chunk_simt(f, s);
    if (e != cudaSuccess) return e;
    // 2. the dS chain
    static bool attr = false;
    if (!attr) {
        if ((e = cudaFuncSetAttribute(bwd_dstate_kernel<Tin, D>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sizeof(DsSmem<D>))) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(bwd_grads_kernel<Tin, D>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sizeof(GrSmem<D>))) != cudaSuccess)
            return e;
        attr = true;
    }
    bwd_dstate_kernel<Tin, D><<<dim3(units, D / DVB), NT, sizeof(DsSmem<D>), s>>>(p, nch, dS_chk);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3. token gradients
    bwd_grads_kernel<Tin, D><<<dim3(nch, units), NT, sizeof(GrSmem<D>), s>>>(p, nch, S_chk, dS_chk);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

size_t chunk_bwd_workspace_bytes(int B, int T, int H, int d) {
    const size_t nch = (size_t)(T + C - 1) / C;
    return 2 * (size_t)B * H * nch * d * d * sizeof(float);
}

cudaError_t launch_chunk_bwd(const BwdProblem &p, cudaStream_t s) {
    if (p.B == 0 || p.T == 0) return cudaSuccess;
    if (p.dtype == 1)
        return p.d == 128 ? launch_bwd_t<__nv_bfloat16, 128>(p, s)
                          : launch_bwd_t<__nv_bfloat16, 64>(p, s);
    return p.d == 128 ? launch_bwd_t<float, 128>(p, s) : launch_bwd_t<float, 64>(p, s);
}

}  // namespace kla
