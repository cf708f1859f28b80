// Curvature-Conditioned Query (CCQ) read-side contraction, "Don't Read
// Everything: A Curvature-Conditioned Query for Linear Attention"
// (gist.science 2606.01294), sections "Derivacao Teorica" and "O Mecanismo":
//
//   Sigma_t   = Cov_{<=t}[k] = M_t / n_t - mu_t mu_t^T,  mu_t = m_t / n_t
//   q_clean_t = (I - lambda_t Sigma_t) q_t
//
// with the running sums M_t = sum_{j<=t} k_j k_j^T, m_t = sum_{j<=t} k_j and
// the count n_t over every key of the sequence up to token t (statistics
// carried across calls like the state).  Section "Integracao": the write rule
// is unchanged and the read is o_t = S_t q_clean_t, so the CCQ layer is the
// KLA forward run on q_clean.
//
// Two passes on the CUDA cores, fp32 arithmetic:
//   ccq_prefix_kernel: per (sequence, head, 16-row block of M) the chunks in
//     order; before adding chunk c it records M (in the input dtype: bf16 for
//     bf16 inputs, whose q_clean is rounded to bf16 anyway, fp32 otherwise)
//     and m (fp32) as the statistics that precede chunk c; at the end the
//     final M, m, n (fp32).
//   ccq_query_kernel: per (chunk, sequence, head), in parallel:
//     y_t = M_prev q_t + sum_{j<=t in chunk} k_j (k_j . q_t)   (= M_t q_t)
//     m_t = m_prev + sum_{j<=t in chunk} k_j,  n_t = n_prev + t + 1
//     q_clean_t = q_t - lambda_t (y_t / n_t - mu_t (mu_t . q_t))

#include <cuda_bf16.h>

#include <cstdint>

#include "kla_internal.h"

namespace kla {
namespace {

constexpr int CC = kChunk;   // 64 tokens per chunk
constexpr int CQ_THREADS = 256;
constexpr int RB = 16;       // rows of M per prefix CTA

__device__ __forceinline__ float ldf(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void stf(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// grid (D / RB, B * H); 256 threads: thread (r = tid / 16, cg = tid % 16)
// owns M[row0 + r][cg + 16 x], x < D/16 (interleaved, so that the 16 lanes
// reading one key row hit 16 banks).
template <typename Tin, int D>
__global__ void __launch_bounds__(CQ_THREADS)
ccq_prefix_kernel(const Tin *__restrict__ k, const float *__restrict__ Ms0,
                  const float *__restrict__ ms0, const float *__restrict__ ns0, int T, int H,
                  int nch, Tin *__restrict__ Mprev, float *__restrict__ mprev,
                  float *__restrict__ Ms_T, float *__restrict__ ms_T, float *__restrict__ ns_T) {
    constexpr int CPT = D / 16;   // columns per thread
    __shared__ float Ks[CC][D + 4];
    const int tid = threadIdx.x, r = tid / 16, cg = tid % 16;
    const int row0 = blockIdx.x * RB, i = row0 + r;
    const long unit = blockIdx.y;
    const long b = unit / H, h = unit % H;
    float acc[CPT];
#pragma unroll
    for (int x = 0; x < CPT; ++x)
        acc[x] = Ms0 ? Ms0[(unit * D + i) * D + cg + 16 * x] : 0.f;
    float msum = 0.f;   // m[row0 + tid] for tid < RB
    if (tid < RB) msum = ms0 ? ms0[unit * D + row0 + tid] : 0.f;
    // chunk keys go through registers: the next chunk's loads are in flight
    // while the current chunk is accumulated
    constexpr int LPT = CC * D / CQ_THREADS;   // key values per thread and chunk
    float pre[LPT];
    auto load_chunk = [&](int cc) {
#pragma unroll
        for (int x = 0; x < LPT; ++x) {
            const int e = tid + x * CQ_THREADS, t = e / D, j = e % D;
            const int tok = cc * CC + t;
            pre[x] = (cc < nch && tok < T) ? ldf(k, (((size_t)b * T + tok) * H + h) * D + j) : 0.f;
        }
    };
    load_chunk(0);
    for (int c = 0; c < nch; ++c) {
        // statistics before chunk c
        Tin *dst = Mprev + (((size_t)unit * nch + c) * D + i) * D + cg;
#pragma unroll
        for (int x = 0; x < CPT; ++x) stf(dst, 16 * x, acc[x]);
        if (tid < RB) mprev[((size_t)unit * nch + c) * D + row0 + tid] = msum;
        __syncthreads();   // previous chunk's keys no longer read
#pragma unroll
        for (int x = 0; x < LPT; ++x) {
            const int e = tid + x * CQ_THREADS;
            Ks[e / D][e % D] = pre[x];
        }
        __syncthreads();
        load_chunk(c + 1);
#pragma unroll 4
        for (int t = 0; t < CC; ++t) {
            const float ki = Ks[t][i];
#pragma unroll
            for (int x = 0; x < CPT; ++x) acc[x] = fmaf(ki, Ks[t][cg + 16 * x], acc[x]);
        }
        if (tid < RB)
            for (int t = 0; t < CC; ++t) msum += Ks[t][row0 + tid];
    }
#pragma unroll
    for (int x = 0; x < CPT; ++x)
        if (Ms_T) Ms_T[(unit * D + i) * D + cg + 16 * x] = acc[x];
    if (tid < RB && ms_T) ms_T[unit * D + row0 + tid] = msum;
    if (blockIdx.x == 0 && tid == 0 && ns_T) ns_T[unit] = (ns0 ? ns0[unit] : 0.f) + (float)T;
}

// grid (nch, B * H); 256 threads: thread (t = tid / 4, ib = tid % 4) owns
// token t of the chunk and dims ib + 4 x, x < D/4 (interleaved, so that the
// four threads of a token read four different banks).
template <typename Tin, int D>
__global__ void __launch_bounds__(CQ_THREADS)
ccq_query_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                 const float *__restrict__ lambda, const float *__restrict__ ns0, int T, int H,
                 int nch, const Tin *__restrict__ Mprev,
                 const float *__restrict__ mprev, Tin *__restrict__ q_clean) {
    constexpr int DPT = D / 4;   // dims per thread
    // rows padded to an odd stride so that lanes walking different rows hit
    // different banks
    constexpr int LD = D + 1;
    extern __shared__ float smq[];
    float *Ks = smq;                 // [CC][LD]
    float *Qs = Ks + CC * LD;        // [CC][LD]
    float *MT = Qs + CC * LD;        // [D][LD], MT[j][i] = M_prev[i][j]
    float *Dm = MT + D * LD;         // [CC][CC + 1]: k_j . q_t for j <= t, else 0
    const int tid = threadIdx.x;
    const int c = blockIdx.x;
    const long unit = blockIdx.y;
    const long b = unit / H, h = unit % H;
    for (int e = tid; e < CC * D; e += CQ_THREADS) {
        const int t = e / D, j = e % D;
        const int tok = c * CC + t;
        const size_t g = (((size_t)b * T + tok) * H + h) * D + j;
        Ks[t * LD + j] = tok < T ? ldf(k, g) : 0.f;
        Qs[t * LD + j] = tok < T ? ldf(q, g) : 0.f;
    }
    const Tin *Mp = Mprev + ((size_t)unit * nch + c) * D * D;
    for (int e = tid; e < D * D; e += CQ_THREADS) {
        const int i = e / D, j = e % D;
        MT[j * LD + i] = ldf(Mp, e);
    }
    __syncthreads();
    for (int e = tid; e < CC * CC; e += CQ_THREADS) {
        const int t = e / CC, j = e % CC;
        float d = 0.f;
        if (j <= t)
            for (int x = 0; x < D; ++x) d = fmaf(Ks[j * LD + x], Qs[t * LD + x], d);
        Dm[t * (CC + 1) + j] = d;
    }
    __syncthreads();

    const int t = tid / 4, ib = tid % 4;
    const int tok = c * CC + t;
    float y[DPT], mc[DPT];
#pragma unroll
    for (int x = 0; x < DPT; ++x) {
        y[x] = 0.f;
        mc[x] = mprev[((size_t)unit * nch + c) * D + ib + 4 * x];
    }
    for (int j = 0; j < D; ++j) {          // M_prev q_t
        const float qj = Qs[t * LD + j];
#pragma unroll
        for (int x = 0; x < DPT; ++x) y[x] = fmaf(MT[j * LD + ib + 4 * x], qj, y[x]);
    }
    for (int j = 0; j < CC; ++j) {         // keys of this chunk up to t (Dm is 0 past t)
        const float d = Dm[t * (CC + 1) + j];
        const float on = j <= t ? 1.f : 0.f;
#pragma unroll
        for (int x = 0; x < DPT; ++x) {
            const float kv = Ks[j * LD + ib + 4 * x];
            y[x] = fmaf(kv, d, y[x]);
            mc[x] = fmaf(kv, on, mc[x]);
        }
    }
    const float n = (ns0 ? ns0[unit] : 0.f) + (float)(c * CC + t + 1);
    const float inv_n = 1.f / n;
    float muq = 0.f;
#pragma unroll
    for (int x = 0; x < DPT; ++x) muq = fmaf(mc[x] * inv_n, Qs[t * LD + ib + 4 * x], muq);
    muq += __shfl_xor_sync(0xffffffffu, muq, 1);
    muq += __shfl_xor_sync(0xffffffffu, muq, 2);
    if (tok < T) {
        const float lam = lambda[((size_t)b * T + tok) * H + h];
        const size_t g = (((size_t)b * T + tok) * H + h) * D + ib;
#pragma unroll
        for (int x = 0; x < DPT; ++x) {
            const float sq = y[x] * inv_n - (mc[x] * inv_n) * muq;
            stf(q_clean, g + 4 * x, Qs[t * LD + ib + 4 * x] - lam * sq);
        }
    }
}

template <typename Tin, int D>
cudaError_t launch_ccq_t(const CcqProblem &p, cudaStream_t s) {
    const int nch = (p.T + CC - 1) / CC;
    const int units = p.B * p.H;
    Tin *Mprev = static_cast<Tin *>(p.ws);
    float *mprev = reinterpret_cast<float *>(static_cast<unsigned char *>(p.ws) +
                                             (size_t)units * nch * D * D * sizeof(Tin));
    ccq_prefix_kernel<Tin, D><<<dim3(D / RB, units), CQ_THREADS, 0, s>>>(
        static_cast<const Tin *>(p.k), p.Ms0, p.ms0, p.ns0, p.T, p.H, nch, Mprev, mprev, p.Ms_T,
        p.ms_T, p.ns_T);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = (size_t)(2 * CC * (D + 1) + D * (D + 1) + CC * (CC + 1)) * sizeof(float);
    static bool attr = false;
    if (!attr) {
        if ((e = cudaFuncSetAttribute(ccq_query_kernel<Tin, D>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
            return e;
        attr = true;
    }
    ccq_query_kernel<Tin, D><<<dim3(nch, units), CQ_THREADS, smem, s>>>(
        static_cast<const Tin *>(p.q), static_cast<const Tin *>(p.k), p.lambda, p.ns0, p.T, p.H,
        nch, Mprev, mprev, static_cast<Tin *>(p.q_clean));
    note_launch();
    return cudaGetLastError();
}

// One token per (b, h) with the statistics updated in place: M += k k^T,
// m += k, n += 1, then q_clean = q - lambda (M q / n - mu (mu . q)).  One CTA
// per (b, h); thread j owns column j of M (M is symmetric, so column j is row
// j): the update and (M q)_j read M[:, j] once and write it once.
template <typename Tin, int D>
__global__ void __launch_bounds__(D)
ccq_step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                const float *__restrict__ lambda, float *__restrict__ Ms, float *__restrict__ ms,
                float *__restrict__ ns, Tin *__restrict__ q_clean) {
    __shared__ float kq[2][D];
    __shared__ float red[D / 32];
    const int j = threadIdx.x;
    const long u = blockIdx.x;
    const float kj = ldf(k, u * D + j), qj = ldf(q, u * D + j);
    kq[0][j] = kj;
    kq[1][j] = qj;
    __syncthreads();
    float *Mu = Ms + (size_t)u * D * D;
    float y = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) {
        const float mij = Mu[(size_t)i * D + j] + kq[0][i] * kj;
        Mu[(size_t)i * D + j] = mij;
        y = fmaf(mij, kq[1][i], y);   // (M q)_j = sum_i M[j][i] q_i, M symmetric
    }
    const float n = ns[u] + 1.f;
    const float mj = ms[u * D + j] + kj;
    ms[u * D + j] = mj;
    float muq = (mj / n) * qj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) muq += __shfl_xor_sync(0xffffffffu, muq, off);
    if ((j & 31) == 0) red[j >> 5] = muq;
    __syncthreads();
    muq = 0.f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) muq += red[w];
    if (j == 0) ns[u] = n;
    stf(q_clean, u * D + j, qj - lambda[u] * (y / n - (mj / n) * muq));
}

template <typename Tin, int D>
cudaError_t launch_step_t(const void *q, const void *k, const float *lambda, float *Ms, float *ms,
                          float *ns, void *q_clean, int BH, cudaStream_t s) {
    ccq_step_kernel<Tin, D><<<BH, D, 0, s>>>(static_cast<const Tin *>(q),
                                              static_cast<const Tin *>(k), lambda, Ms, ms, ns,
                                              static_cast<Tin *>(q_clean));
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ccq_step(const void *q, const void *k, const float *lambda, float *Ms,
                            float *ms, float *ns, void *q_clean, int BH, int d, int dtype,
                            cudaStream_t s) {
    if (BH == 0) return cudaSuccess;
    if (dtype == 1)
        return d == 128 ? launch_step_t<__nv_bfloat16, 128>(q, k, lambda, Ms, ms, ns, q_clean, BH, s)
                        : launch_step_t<__nv_bfloat16, 64>(q, k, lambda, Ms, ms, ns, q_clean, BH, s);
    return d == 128 ? launch_step_t<float, 128>(q, k, lambda, Ms, ms, ns, q_clean, BH, s)
                    : launch_step_t<float, 64>(q, k, lambda, Ms, ms, ns, q_clean, BH, s);
}

size_t ccq_workspace_bytes(int B, int T, int H, int d, int dtype) {
    const size_t nch = (size_t)(T + CC - 1) / CC;
    const size_t es = dtype == 1 ? 2 : 4;
    return (size_t)B * H * nch * ((size_t)d * d * es + (size_t)d * 4);
}

cudaError_t launch_ccq(const CcqProblem &p, cudaStream_t s) {
    if (p.B == 0 || p.T == 0) return cudaSuccess;
    if (p.dtype == 1)
        return p.d == 128 ? launch_ccq_t<__nv_bfloat16, 128>(p, s)
                          : launch_ccq_t<__nv_bfloat16, 64>(p, s);
    return p.d == 128 ? launch_ccq_t<float, 128>(p, s) : launch_ccq_t<float, 64>(p, s);
}

}  // namespace kla
