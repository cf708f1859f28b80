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
// bf16 inputs with d = 128 take the tensor cores: y_t = M_t q_t is a gated
// delta-rule product with no decay whose chunk write is K^T K, so the chunked
// tcgen05 forward runs it in its CCQ mode (W = 0, U~ = K: the state pass
// gives y = Q M_prev + lower(Q K^T) K and carries M); then
// whose first phase also writes the sum of each chunk's keys; then
//   ccq_finish_kernel: per (chunk, sequence, head) m_prev from those sums, the
//     running key sum m_t inside the chunk, n_t, mu_t . q_t and q_clean_t.
//
// Other inputs: two passes on the CUDA cores, fp32 arithmetic:
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

// ---- tensor-core path (bf16, D = 128) ----
constexpr int TD = 128;

__device__ __forceinline__ void unpack8(const uint4 v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

// grid (nch, B * H); 256 threads, three CTAs per SM.  Every load is issued up
// front: q and y rows of the chunk go to shared memory by asynchronous copies
// (16-byte piece pc of token row t at position pc ^ 4 (t & 1), so that the
// two tokens read by eight consecutive lanes fall in different banks), the
// keys through registers into an fp32 tile, and half of the key sums of the
// preceding chunks for feature tid % 128 into registers.  Thread j < 128 then
// turns key column j into the running sums m_t (from m before the chunk), and
// thread (t = tid / 4, part = tid % 4) finishes token t on the pieces part +
// 4 x.
constexpr int FK_LD = TD + 4;   // fp32 key row stride: 16-byte aligned rows
constexpr size_t FK_SMEM = (size_t)CC * FK_LD * 4 + 2 * (size_t)CC * TD * 2 + 2 * TD * 4;

__global__ void __launch_bounds__(CQ_THREADS, 3)
ccq_finish_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                  const __nv_bfloat16 *__restrict__ y, const float *__restrict__ lambda,
                  const float *__restrict__ ms0, const float *__restrict__ ns0,
                  const float *__restrict__ csum, int T, int H, int nch,
                  __nv_bfloat16 *__restrict__ q_clean, float *__restrict__ ms_T,
                  float *__restrict__ ns_T) {
    extern __shared__ __align__(16) unsigned char fsm[];
    float *Ks = reinterpret_cast<float *>(fsm);                        // [CC][FK_LD]
    unsigned char *Qs = fsm + (size_t)CC * FK_LD * 4;                  // [CC][256 B]
    unsigned char *Ys = Qs + (size_t)CC * TD * 2;                      // [CC][256 B]
    float *mp = reinterpret_cast<float *>(Ys + (size_t)CC * TD * 2);   // [2][TD]
    const int tid = threadIdx.x, c = blockIdx.x;
    const long unit = blockIdx.y, b = unit / H, h = unit % H;
    const size_t tok_stride = (size_t)H * TD;
    const size_t base = ((size_t)b * T * H + h) * TD;   // token 0 of (b, h)

    // piece e of the chunk: token e / 16, 16-byte piece e % 16
    uint4 ka[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int e = tid + x * CQ_THREADS, te = e >> 4, pc = e & 15, kt = c * CC + te;
        if (kt < T) {
            const size_t o = base + (size_t)kt * tok_stride + pc * 8;
            const int pos = te * 256 + ((pc ^ ((te & 1) << 2)) << 4);
            cp_async16(Qs + pos, q + o);
            cp_async16(Ys + pos, y + o);
            ka[x] = *reinterpret_cast<const uint4 *>(k + o);
        } else {
            ka[x] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    // m before the chunk: the initial sum plus the preceding chunks' sums,
    // chunks cc = half, half + 2, ... for this thread
    const int j = tid & (TD - 1), half = tid >> 7;
    const float *cs = csum + ((size_t)b * nch * H + h) * TD + j;   // chunk cc at cc * H * TD
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int cc = half;
    for (; cc + 6 < c; cc += 8) {
        a0 += cs[(size_t)cc * H * TD];
        a1 += cs[(size_t)(cc + 2) * H * TD];
        a2 += cs[(size_t)(cc + 4) * H * TD];
        a3 += cs[(size_t)(cc + 6) * H * TD];
    }
    for (; cc < c; cc += 2) a0 += cs[(size_t)cc * H * TD];
    mp[half * TD + j] = (a0 + a1) + (a2 + a3) + (half == 0 && ms0 ? ms0[unit * TD + j] : 0.f);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int e = tid + x * CQ_THREADS;
        float f[8];
        unpack8(ka[x], f);
        float4 *dst = reinterpret_cast<float4 *>(Ks + (e >> 4) * FK_LD + (e & 15) * 8);
        dst[0] = make_float4(f[0], f[1], f[2], f[3]);
        dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    const int t = tid >> 2, part = tid & 3, tok = c * CC + t;
    const bool live = tok < T;
    const float lam = live ? lambda[((size_t)b * T + tok) * H + h] : 0.f;
    const float n0 = ns0 ? ns0[unit] : 0.f;
    __syncthreads();
    if (tid < TD) {
        float run = mp[tid] + mp[TD + tid];
#pragma unroll
        for (int t0 = 0; t0 < CC; t0 += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = Ks[(t0 + i) * FK_LD + tid];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                run += v[i];
                Ks[(t0 + i) * FK_LD + tid] = run;
            }
        }
        if (c == nch - 1 && ms_T) ms_T[unit * TD + tid] = run;
    }
    if (c == nch - 1 && tid == 0 && ns_T) ns_T[unit] = n0 + (float)T;
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    __syncthreads();

    const float inv_n = 1.f / (n0 + (float)(c * CC + t + 1));
    const float *mrow = Ks + t * FK_LD;
    const int sw = (t & 1) << 2;
    float muq = 0.f;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int pc = part + 4 * x;
        float qf[8];
        unpack8(*reinterpret_cast<const uint4 *>(Qs + t * 256 + ((pc ^ sw) << 4)), qf);
        const float4 m0 = *reinterpret_cast<const float4 *>(mrow + pc * 8);
        const float4 m1 = *reinterpret_cast<const float4 *>(mrow + pc * 8 + 4);
        muq = fmaf(m0.x, qf[0], muq); muq = fmaf(m0.y, qf[1], muq);
        muq = fmaf(m0.z, qf[2], muq); muq = fmaf(m0.w, qf[3], muq);
        muq = fmaf(m1.x, qf[4], muq); muq = fmaf(m1.y, qf[5], muq);
        muq = fmaf(m1.z, qf[6], muq); muq = fmaf(m1.w, qf[7], muq);
    }
    muq *= inv_n;   // mu_t . q_t
    muq += __shfl_xor_sync(0xffffffffu, muq, 1);
    muq += __shfl_xor_sync(0xffffffffu, muq, 2);
    if (live) {
        const size_t o0 = base + (size_t)tok * tok_stride;
        const float mscale = inv_n * muq;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int pc = part + 4 * x;
            float qf[8], yf[8], mf[8];
            unpack8(*reinterpret_cast<const uint4 *>(Qs + t * 256 + ((pc ^ sw) << 4)), qf);
            unpack8(*reinterpret_cast<const uint4 *>(Ys + t * 256 + ((pc ^ sw) << 4)), yf);
            const float4 m0 = *reinterpret_cast<const float4 *>(mrow + pc * 8);
            const float4 m1 = *reinterpret_cast<const float4 *>(mrow + pc * 8 + 4);
            mf[0] = m0.x; mf[1] = m0.y; mf[2] = m0.z; mf[3] = m0.w;
            mf[4] = m1.x; mf[5] = m1.y; mf[6] = m1.z; mf[7] = m1.w;
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const float c0 = yf[i] * inv_n - mf[i] * mscale;
                const float c1 = yf[i + 1] * inv_n - mf[i + 1] * mscale;
                const __nv_bfloat162 o2 = __floats2bfloat162_rn(qf[i] - lam * c0,
                                                                qf[i + 1] - lam * c1);
                w[i / 2] = *reinterpret_cast<const uint32_t *>(&o2);
            }
            *reinterpret_cast<uint4 *>(q_clean + o0 + pc * 8) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool ccq_use_tc(int B, int T, int d, int dtype) {
    return chunk_tc_supported(d, dtype) && (long)B * T >= CC;
}

// Tensor-core workspace after the header: the chunked forward's workspace,
// y [B, T, H, 128] bf16, the chunk key sums [B, nch, H, 128] fp32.
struct CcqTcLayout {
    size_t tc, y, csum, total;
};
CcqTcLayout ccq_tc_layout(int B, int T, int H) {
    const long nch = (T + CC - 1) / CC;
    CcqTcLayout L;
    L.tc = 0;
    L.y = align_up(chunk_tc_workspace_bytes((long)B * nch, H, B), 256);
    L.csum = align_up(L.y + (size_t)B * T * H * TD * 2, 256);
    L.total = L.csum + (size_t)B * H * nch * TD * 4;
    return L;
}

cudaError_t launch_ccq_tc(const CcqProblem &p, cudaStream_t s) {
    const int nch = (p.T + CC - 1) / CC;
    const CcqTcLayout L = ccq_tc_layout(p.B, p.T, p.H);
    unsigned char *ws = static_cast<unsigned char *>(p.ws) + kWsHeader;
    __nv_bfloat16 *yb = reinterpret_cast<__nv_bfloat16 *>(ws + L.y);
    float *csum = reinterpret_cast<float *>(ws + L.csum);
    // y = M_t q_t on the tensor cores: the chunked forward in its CCQ mode,
    // with the statistics M as its state (v = k feeds only the unused V tile;
    // eta, here lambda, is read but does not enter)
    Problem f{};
    f.q = p.q; f.k = p.k; f.v = p.k;
    f.alpha = nullptr; f.eta = p.lambda; f.eps = 0.f;
    f.S0 = p.Ms0; f.S_T = p.Ms_T; f.o = yb;
    f.cu_seqlens = nullptr;
    f.n_seq = p.B; f.T = p.T; f.total_T = p.B * p.T; f.H = p.H; f.d = TD; f.dtype = p.dtype;
    f.beta_mode = 1; f.mode = 1; f.csum = csum;
    f.status = static_cast<unsigned *>(p.ws);
    f.ws = ws + L.tc;
    f.ws_bytes = L.y - L.tc;
    const long nchunks = (long)p.B * nch;
    cudaError_t e = cudaMemsetAsync(p.ws, 0, kWsHeader + chunk_tc_reset_bytes(f, nchunks), s);
    if (e != cudaSuccess) return e;
    if ((e = launch_chunk_tc(f, nchunks, s)) != cudaSuccess) return e;
    static bool fattr = false;
    if (!fattr) {
        if ((e = cudaFuncSetAttribute(ccq_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)FK_SMEM)) != cudaSuccess)
            return e;
        fattr = true;
    }
    const dim3 grid(nch, p.B * p.H);
    ccq_finish_kernel<<<grid, CQ_THREADS, FK_SMEM, s>>>(
        static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k), yb,
        p.lambda, p.ms0, p.ns0, csum, p.T, p.H, nch, static_cast<__nv_bfloat16 *>(p.q_clean),
        p.ms_T, p.ns_T);
    note_launch();
    return cudaGetLastError();
}

// ---- CUDA-core path ----
template <typename Tin, int D>
cudaError_t launch_ccq_t(const CcqProblem &p, cudaStream_t s) {
    const int nch = (p.T + CC - 1) / CC;
    const int units = p.B * p.H;
    cudaError_t e0 = cudaMemsetAsync(p.ws, 0, sizeof(unsigned), s);   // status word
    if (e0 != cudaSuccess) return e0;
    Tin *Mprev = reinterpret_cast<Tin *>(static_cast<unsigned char *>(p.ws) + kWsHeader);
    float *mprev = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(Mprev) +
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
    if (ccq_use_tc(B, T, d, dtype)) return kWsHeader + ccq_tc_layout(B, T, H).total;
    const size_t nch = (size_t)(T + CC - 1) / CC;
    const size_t es = dtype == 1 ? 2 : 4;
    return kWsHeader + (size_t)B * H * nch * ((size_t)d * d * es + (size_t)d * 4);
}

cudaError_t launch_ccq(const CcqProblem &p, cudaStream_t s) {
    if (p.B == 0 || p.T == 0) return cudaSuccess;
    if (ccq_use_tc(p.B, p.T, p.d, p.dtype)) return launch_ccq_tc(p, s);
    if (p.dtype == 1)
        return p.d == 128 ? launch_ccq_t<__nv_bfloat16, 128>(p, s)
                          : launch_ccq_t<__nv_bfloat16, 64>(p, s);
    return p.d == 128 ? launch_ccq_t<float, 128>(p, s) : launch_ccq_t<float, 64>(p, s);
}

}  // namespace kla
