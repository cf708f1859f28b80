// Chunkwise-parallel KLA prefill on CUDA cores, fp32 arithmetic.
//
// This is the exact-precision path (fp32 inputs) and covers every supported
// size and dtype.  The algorithm is Gated DeltaNet's blockwise solver with
// the Kaczmarz coefficients on the diagonal (Kaczmarz Linear Attention
// summary, gist.science 2605.08587, sections "Implementacao" and
// "A Regra de Atualizacao KLA": B = Diag(beta_1..beta_C) is the only change).
// For one chunk of C = 64 tokens starting from state S (dk x dv):
//
//   g_t    = sum_{s<=t} log alpha_s          Gamma_ts = exp(g_t - g_s), s <= t
//   beta_t = eta_t / (||k_t||^2 + eps)
//   A_kk   = strict_lower(beta_t Gamma_ts k_t.k_s)
//   A_qk   = lower(Gamma_ts q_t.k_s)
//   T      = (I + A_kk)^{-1}                 (forward substitution)
//   U      = T diag(beta) (V - diag(exp g) K S)
//   O      = diag(exp g) Q S + A_qk U
//   S'     = exp(g_C) S + K^T diag(exp(g_C - g)) U
//
// One CTA owns one (sequence, head) and a 32-column block of dv; it walks
// the chunks of its sequence in order, keeping its state block in shared
// memory.  Tail positions of a partial chunk are masked as identity tokens
// (k = q = v = 0, alpha = 1, beta = 0).

#include <cuda_bf16.h>

#include "kla_internal.h"
#include "kla_simt_inverse.cuh"
#include "kla_simt_tile.cuh"

namespace kla {
namespace {

constexpr int C = kChunk;
constexpr int DVB = 32;          // dv columns per CTA
constexpr int NT = 256;          // threads per CTA

__device__ __forceinline__ void st_out(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

template <int D>
struct Smem {
    float K[C][D + 1];
    float Q[C][D + 1];
    float V[C][DVB + 1];
    float Akk[C][C + 1];
    float Tm[C][C + 1];
    float Aqk[C][C + 1];
    float S[D][DVB + 1];
    float KS[C][DVB + 1];
    float QS[C][DVB + 1];
    float R[C][DVB + 1];
    float U[C][DVB + 1];
    float alpha[C], eta[C], g[C], beta[C], eg[C], egc[C];
};

template <typename Tin, int D>
__global__ void __launch_bounds__(NT, 1) chunk_simt_kernel(Problem p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem<D> &sm = *reinterpret_cast<Smem<D> *>(smem_raw);

    const int tid = threadIdx.x;
    const int unit = blockIdx.x;
    const int seq = unit / p.H, h = unit % p.H;
    const int jb = blockIdx.y * DVB;
    const int H = p.H;

    if (p.status != nullptr && *(volatile unsigned *)p.status != kDevOk) return;

    long start, len;
    if (p.cu_seqlens) {
        start = p.cu_seqlens[seq];
        const long end = p.cu_seqlens[seq + 1];
        len = end - start;
        if (start < 0 || len < 0 || end > p.total_T) return;  // rejected by the check kernel
    } else {
        start = (long)seq * p.T;
        len = p.T;
    }

    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    Tin *o = static_cast<Tin *>(p.o);
    const size_t sbase = ((size_t)seq * H + h) * D * D;

    for (int x = tid; x < D * DVB; x += NT) {
        const int i = x / DVB, j = x % DVB;
        sm.S[i][j] = p.S0 ? p.S0[sbase + (size_t)i * D + jb + j] : 0.f;
    }

    // first chunk of this sequence in the chunk-slot numbering of the
    // recorded states (slot = chunk * H + head)
    const long chunk0 =
        p.cu_seqlens ? (p.chunk_prefix ? p.chunk_prefix[seq] : 0) : (long)seq * ((p.T + C - 1) / C);
    for (long c0 = 0; c0 < len; c0 += C) {
        const int nc = (int)min((long)C, len - c0);
        __syncthreads();  // previous chunk finished with K, Q, V, S
        if (p.S_chk) {    // the state at the chunk's start, for the backward pass
            float *dst = static_cast<float *>(p.S_chk) + ((size_t)(chunk0 + c0 / C) * H + h) * D * D;
            for (int x = tid; x < D * DVB; x += NT) {
                const int i = x / DVB, j = x % DVB;
                dst[(size_t)i * D + jb + j] = sm.S[i][j];
            }
        }

        // ---- load the chunk (masked tail = identity tokens) ----
        load_tile<Tin, C, D, D + 1, NT>(&sm.K[0][0], k, start + c0, nc, H, h, D, 0, tid);
        load_tile<Tin, C, D, D + 1, NT>(&sm.Q[0][0], q, start + c0, nc, H, h, D, 0, tid);
        load_tile<Tin, C, DVB, DVB + 1, NT>(&sm.V[0][0], v, start + c0, nc, H, h, D, jb, tid);
        if (tid < C) {
            const bool ok = tid < nc;
            const size_t row = (size_t)(start + c0 + tid) * H + h;
            sm.alpha[tid] = (ok && p.alpha) ? p.alpha[row] : 1.f;
            sm.eta[tid] = ok ? p.eta[row] : 0.f;
        }
        __syncthreads();

        // ---- beta from the key norms; log-decay prefix sums ----
        if (tid < C) {
            float n2 = 0.f;
            for (int i = 0; i < D; ++i) n2 = fmaf(sm.K[tid][i], sm.K[tid][i], n2);
            const float den = n2 + p.eps;
            const float b = p.beta_mode ? sm.eta[tid] : (den != 0.f ? sm.eta[tid] / den : 0.f);
            sm.beta[tid] = tid < nc ? b : 0.f;
        } else if (tid < C + 32) {
            // warp 2: inclusive scan of log alpha over 64 positions, in double
            const int lane = tid - C;
            double a0 = (double)logf(sm.alpha[lane]);
            double a1 = (double)logf(sm.alpha[lane + 32]);
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double u0 = __shfl_up_sync(0xffffffffu, a0, off);
                const double u1 = __shfl_up_sync(0xffffffffu, a1, off);
                if (lane >= off) { a0 += u0; a1 += u1; }
            }
            const double tot0 = __shfl_sync(0xffffffffu, a0, 31);
            a1 += tot0;
            sm.g[lane] = (float)a0;
            sm.g[lane + 32] = (float)a1;
            const double gC = __shfl_sync(0xffffffffu, a1, 31);
            sm.eg[lane] = (float)exp(a0);
            sm.eg[lane + 32] = (float)exp(a1);
            sm.egc[lane] = (float)exp(gC - a0);
            sm.egc[lane + 32] = (float)exp(gC - a1);
        }
        __syncthreads();

        // ---- Gram products A_kk (strict lower, beta rows) and A_qk (lower) ----
        {
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
                        kt[m] = sm.K[bt * 4 + m][i];
                        qt[m] = sm.Q[bt * 4 + m][i];
                        ks[m] = sm.K[bs * 4 + m][i];
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
                    const float gam = (s <= t) ? expf(sm.g[t] - sm.g[s]) : 0.f;
                    sm.Akk[t][s] = (s < t) ? sm.beta[t] * gam * akk[m][n] : 0.f;
                    sm.Aqk[t][s] = (s <= t) ? gam * aqk[m][n] : 0.f;
                }
        }
        __syncthreads();

        // ---- T = (I + A_kk)^{-1} (blocked; U is its scratch); K S and Q S ----
        invert_unit_lower64(sm.Akk, sm.Tm, &sm.U[0][0], tid);
        {
            const int t = tid / 4, jq = (tid % 4) * 8;
            float ks[8], qs[8];
#pragma unroll
            for (int n = 0; n < 8; ++n) ks[n] = qs[n] = 0.f;
            for (int i = 0; i < D; ++i) {
                const float kti = sm.K[t][i], qti = sm.Q[t][i];
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    const float s_ = sm.S[i][jq + n];
                    ks[n] = fmaf(kti, s_, ks[n]);
                    qs[n] = fmaf(qti, s_, qs[n]);
                }
            }
            const float bt = sm.beta[t], egt = sm.eg[t];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                sm.R[t][jq + n] = bt * (sm.V[t][jq + n] - egt * ks[n]);
                sm.QS[t][jq + n] = egt * qs[n];
            }
        }
        __syncthreads();

        // ---- U = T R ----
        {
            const int t = tid / 4, jq = (tid % 4) * 8;
            float u[8];
#pragma unroll
            for (int n = 0; n < 8; ++n) u[n] = 0.f;
            for (int s = 0; s <= t; ++s) {
                const float tts = sm.Tm[t][s];
#pragma unroll
                for (int n = 0; n < 8; ++n) u[n] = fmaf(tts, sm.R[s][jq + n], u[n]);
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) sm.U[t][jq + n] = u[n];
        }
        __syncthreads();

        // ---- O = diag(exp g) Q S + A_qk U ;  S' = exp(g_C) S + K^T diag(exp(g_C-g)) U ----
        {
            const int t = tid / 4, jq = (tid % 4) * 8;
            float acc[8];
#pragma unroll
            for (int n = 0; n < 8; ++n) acc[n] = sm.QS[t][jq + n];
            for (int s = 0; s <= t; ++s) {
                const float a = sm.Aqk[t][s];
#pragma unroll
                for (int n = 0; n < 8; ++n) acc[n] = fmaf(a, sm.U[s][jq + n], acc[n]);
            }
            if (o && t < nc) {
                const size_t row = (size_t)(start + c0 + t) * H + h;
#pragma unroll
                for (int n = 0; n < 8; ++n) st_out(o, row * D + jb + jq + n, acc[n]);
            }
        }
        {
            constexpr int TPR = NT / D;          // threads per state row
            constexpr int JPT = DVB / TPR;       // columns per thread
            const int i = tid / TPR, j0 = (tid % TPR) * JPT;
            const float egC = sm.eg[C - 1];
            float acc[JPT];
#pragma unroll
            for (int n = 0; n < JPT; ++n) acc[n] = egC * sm.S[i][j0 + n];
            for (int t = 0; t < nc; ++t) {
                const float kw = sm.K[t][i] * sm.egc[t];
#pragma unroll
                for (int n = 0; n < JPT; ++n) acc[n] = fmaf(kw, sm.U[t][j0 + n], acc[n]);
            }
#pragma unroll
            for (int n = 0; n < JPT; ++n) sm.S[i][j0 + n] = acc[n];
        }
    }
    __syncthreads();

    if (p.S_T) {
        for (int x = tid; x < D * DVB; x += NT) {
            const int i = x / DVB, j = x % DVB;
            p.S_T[sbase + (size_t)i * D + jb + j] = sm.S[i][j];
        }
    }
}

template <typename Tin, int D>
cudaError_t launch_t(const Problem &p, cudaStream_t s) {
    const size_t smem = sizeof(Smem<D>);
    cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<Tin, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_seq * p.H, D / DVB);
    chunk_simt_kernel<Tin, D><<<grid, NT, smem, s>>>(p);
    note_launch();
    return cudaGetLastError();
}

// Validates cu_seqlens on the device: cu[0] == 0, non-decreasing,
// cu[N] == total_T.  Writes the verdict into the workspace status word, which
// every later kernel of the same call reads before touching memory.
__global__ void check_seqlens_kernel(const int *cu, int N, int total_T, unsigned *status) {
    __shared__ int bad;
    if (threadIdx.x == 0) bad = (cu[0] != 0 || cu[N] != total_T) ? 1 : 0;
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x)
        if (cu[i + 1] < cu[i]) atomicOr(&bad, 1);
    __syncthreads();
    if (threadIdx.x == 0) *status = bad ? (unsigned)kDevBadSeqlens : (unsigned)kDevOk;
}

}  // namespace

cudaError_t launch_check_seqlens(const Problem &p, cudaStream_t s) {
    check_seqlens_kernel<<<1, 256, 0, s>>>(p.cu_seqlens, p.n_seq, p.total_T, p.status);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_chunk_simt(const Problem &p, cudaStream_t s) {
    if (p.n_seq == 0) return cudaSuccess;
    if (p.dtype == 1) {
        if (p.d == 128) return launch_t<__nv_bfloat16, 128>(p, s);
        return launch_t<__nv_bfloat16, 64>(p, s);
    }
    if (p.d == 128) return launch_t<float, 128>(p, s);
    return launch_t<float, 64>(p, s);
}

}  // namespace kla
