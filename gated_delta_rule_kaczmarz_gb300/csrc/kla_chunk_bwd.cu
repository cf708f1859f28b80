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
#include "kla_simt_inverse.cuh"
#include "kla_simt_tile.cuh"
#include "kla_tc.cuh"
#include "kla_tmap.h"

namespace kla {
namespace {

constexpr int C = kChunk;
constexpr int NT = 256;
constexpr int DVB = 32;   // dv columns per CTA of the state-gradient chain


// Per-chunk vectors.  Tail positions of a partial chunk are identity tokens
// (k = q = v = 0, alpha = 1, eta = 0, beta = 0).
struct Vec {
    float alpha[C], eta[C], g[C], beta[C], eg[C], egc[C], den[C];
};

// Token rows and chunks of sequence n: fixed length (rows n T .. n T + T - 1,
// chunks n nch ..) or packed varlen (cu_seqlens, chunk_prefix).  Recorded
// states are indexed by chunk slot = chunk * H + head.
struct SeqGeo {
    long start, chunk0;
    int len, nch;
};
__device__ __forceinline__ SeqGeo seq_geo(const BwdProblem &p, int n) {
    SeqGeo g;
    if (p.cu_seqlens) {
        g.start = p.cu_seqlens[n];
        g.len = p.cu_seqlens[n + 1] - p.cu_seqlens[n];
        g.chunk0 = p.chunk_prefix[n];
    } else {
        g.start = (long)n * p.T;
        g.len = p.T;
        g.chunk0 = (long)n * ((p.T + C - 1) / C);
    }
    g.nch = (g.len + C - 1) / C;
    return g;
}

template <typename Tin, int D>
__device__ void load_kq(float (*K)[D + 1], float (*Q)[D + 1], Vec &v, const BwdProblem &p,
                        long row0, int nc, int h, int tid) {
    load_tile<Tin, C, D, D + 1, NT>(&K[0][0], static_cast<const Tin *>(p.k), row0, nc, p.H, h, D,
                                    0, tid);
    load_tile<Tin, C, D, D + 1, NT>(&Q[0][0], static_cast<const Tin *>(p.q), row0, nc, p.H, h, D,
                                    0, tid);
    if (tid < C) {
        const bool ok = tid < nc;
        const size_t r = (size_t)(row0 + tid) * p.H + h;
        v.alpha[tid] = (ok && p.alpha) ? p.alpha[r] : 1.f;
        v.eta[tid] = ok ? p.eta[r] : 0.f;
    }
}

// beta, ||k||^2 + eps and the in-chunk log-decay prefix sums (after K, alpha
// and eta are in shared memory).
template <int D, int LK = D + 1>
__device__ void chunk_vectors(const float (*K)[LK], Vec &v, float eps, int beta_mode, int nc,
                              int tid) {
    if (tid < C) {
        float n2 = 0.f;
        if constexpr (LK % 4 == 0) {
            for (int i = 0; i < D; i += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&K[tid][i]);
                n2 = fmaf(k4.x, k4.x, n2); n2 = fmaf(k4.y, k4.y, n2);
                n2 = fmaf(k4.z, k4.z, n2); n2 = fmaf(k4.w, k4.w, n2);
            }
        } else {
            for (int i = 0; i < D; ++i) n2 = fmaf(K[tid][i], K[tid][i], n2);
        }
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
template <int D, bool kApply, int LK = D + 1, int LM = C + 1>
__device__ void gram(const float (*K)[LK], const float (*Q)[LK], const Vec &v,
                     float (*Mkk)[LM], float (*Mqk)[LM], int tid) {
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
__global__ void __launch_bounds__(NT, 1) bwd_dstate_kernel(BwdProblem p, float *dS_chk) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    DsSmem<D> &sm = *reinterpret_cast<DsSmem<D> *>(smem_raw);
    const int tid = threadIdx.x;
    const int unit = blockIdx.x, h = unit % p.H;
    const int jb = blockIdx.y * DVB;
    if (p.status != nullptr && *(volatile unsigned *)p.status != kDevOk) return;
    const SeqGeo sg = seq_geo(p, unit / p.H);
    const Tin *dout = static_cast<const Tin *>(p.dout);
    const size_t sbase = (size_t)unit * D * D;

    for (int x = tid; x < D * DVB; x += NT) {
        const int i = x / DVB, j = x % DVB;
        sm.dS[i][j] = p.dS_T ? p.dS_T[sbase + (size_t)i * D + jb + j] : 0.f;
    }
    for (int c = sg.nch - 1; c >= 0; --c) {
        const long row0 = sg.start + (long)c * C;
        const int nc = min(C, sg.len - c * C);
        __syncthreads();   // the previous chunk is done with every tile
        float *rec = dS_chk + ((size_t)(sg.chunk0 + c) * p.H + h) * D * D;   // dS' of chunk c
        for (int x = tid; x < D * DVB; x += NT) {
            const int i = x / DVB, j = x % DVB;
            rec[(size_t)i * D + jb + j] = sm.dS[i][j];
        }
        load_kq<Tin, D>(sm.K, sm.Q, sm.v, p, row0, nc, h, tid);
        load_tile<Tin, C, DVB, DVB + 1, NT>(&sm.dO[0][0], dout, row0, nc, p.H, h, D, jb, tid);
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
        invert_unit_lower64(sm.Akk, sm.Tm, &sm.dR[0][0], tid);
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

// dS chain for bf16, d = 128 on the tensor cores, from the tensor-core
// forward's chunk workspace: W = T diag(beta exp g) K (bf16), A^T (bf16,
// row = key, column = query) and g of every chunk, so that the chain needs no
// Gram product and no inverse:
//   dU = A_qk^T dO + diag(exp(g_C - g)) K dS'
//   dS = exp(g_C) dS' + Q^T diag(exp g) dO - W^T dU
// One CTA per (sequence, head), transposed so that the 128 value columns j of
// dS are the rows of every product (one per TMEM lane):
//   X = dS'^T K^T,  Y = dO^T A_qk            (128 x 64: column t a token)
//   dU^T = X diag(exp(g_C - g)) + Y          (bf16 into TMEM: an MMA operand)
//   D = dO^T diag(exp g) Q - dU^T W          (128 x 128)
//   dS^T <- exp(g_C) dS'^T + D               (fp32 registers)
// The serial chain per chunk is X -> dU -> D -> dS'; Y and the Q half of D
// depend on the chunk's inputs only and are issued ahead.  A loader warp
// brings each chunk's K, Q, dO (token rows), W and A^T (workspace) by TMA,
// two chunks in flight; an MMA warp issues the products; eight main warps
// hold the state, thread (lane j, half hf) the columns i in [64 hf, 64 hf + 64)
// of row j of dS^T (so that dS0's rows, fixed i, are written by
// a warp as 32 consecutive floats), and dS' of every chunk is recorded as
// the bf16 dS'^T tile that feeds X (a bulk copy of shared memory).
namespace dtc {
constexpr int D = 128;
constexpr int NS = 2;                                // stages
constexpr uint32_t T64 = 64u * 128u;                 // 64 rows x 64 bf16 (one slab)
constexpr uint32_t ST_K = 0, ST_Q = 2 * T64, ST_O = 4 * T64, ST_W = 6 * T64, ST_A = 8 * T64;
constexpr uint32_t ST_BYTES = 9 * T64;               // K, Q, dO, W (two slabs each), A^T
constexpr uint32_t ST_TX = ST_BYTES;                 // + g (bulk copy, 256 B)
constexpr uint32_t SM_S = NS * ST_BYTES;             // dS'^T (bf16, 128 x 128, K-major)
constexpr uint32_t SM_G = SM_S + 2 * 128u * 128u;    // g of each stage [NS][64]
constexpr uint32_t SM_E = SM_G + NS * 256;           // exp g, exp(g_C - g) of each stage [NS][2][64]
constexpr uint32_t SMEM = SM_E + NS * 512 + 1024;
constexpr int NMAIN = 8, THREADS = (NMAIN + 2) * 32;
constexpr uint32_t TM_X = 0, TM_Y = 64, TM_U = 128, TM_D = 256;   // D: two buffers of 128
static_assert(SMEM <= 232448, "dS chain shared memory");
}  // namespace dtc

__device__ __forceinline__ unsigned char *dtc_align1024(unsigned char *p) {
    const uint32_t a = tc::smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}
__device__ __forceinline__ uint32_t dtc_pack(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);   // a -> low half
    return *reinterpret_cast<const uint32_t *>(&v);
}

__global__ void __launch_bounds__(dtc::THREADS, 1)
bwd_dstate_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mo, const __grid_constant__ CUtensorMap mw,
                     const __grid_constant__ CUtensorMap ma, BwdProblem p, unsigned char *dS_img,
                     const float *g_ws) {
    using namespace dtc;
    using namespace tc;
    extern __shared__ unsigned char dtc_smem[];
    unsigned char *sm = dtc_align1024(dtc_smem);
    __shared__ uint64_t bar_ld[NS], bar_empty[NS];
    __shared__ uint64_t bar_prep, bar_s, bar_x, bar_u, bar_d, bar_fin;
    __shared__ uint32_t tslot;
    __shared__ int sAbort;
    unsigned char *sS = sm + SM_S;
    float *sg = reinterpret_cast<float *>(sm + SM_G);
    float *se = reinterpret_cast<float *>(sm + SM_E);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, h = unit % p.H;
    const SeqGeo geo = seq_geo(p, unit / p.H);
    const int nch = geo.nch;
    const size_t sbase = (size_t)unit * D * D;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_ld[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_prep, NMAIN);
        mbar_init(&bar_s, NMAIN);
        mbar_init(&bar_x, 1);
        mbar_init(&bar_u, NMAIN);
        mbar_init(&bar_d, 1);
        mbar_init(&bar_fin, 1);
        fence_mbar_init();
        sAbort = (p.status != nullptr && *(volatile const unsigned *)p.status != kDevOk) ? 1 : 0;
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tslot;
    const int pre_abort = sAbort;   // read by every thread before any can change it
    __syncthreads();
    if (pre_abort) {
        if (warp == 0) tmem_dealloc(tb, 512);
        return;
    }
    auto fail = [&]() {
        *(volatile int *)&sAbort = 1;
        if (p.status) atomicCAS(p.status, 0u, kDevTimeout);
    };
    // step k handles chunk nch - 1 - k
    auto slot_of = [&](int k) { return (geo.chunk0 + (nch - 1 - k)) * p.H + h; };

    if (warp == NMAIN + 1) {
        // ------------------------------------------------------------ loader
        int k = 0;
        for (; k < nch; ++k) {
            const int s = k % NS, r = k / NS;
            if (r >= 1 &&
                !__all_sync(0xffffffffu,
                            mbar_wait_or_abort(&bar_empty[s], (uint32_t)((r - 1) & 1), &sAbort))) {
                fail();
                break;
            }
            if (lane == 0) {
                unsigned char *st = sm + s * ST_BYTES;
                const int c = nch - 1 - k;
                const int row0 = (int)(geo.start + (long)c * C);
                const long slot = slot_of(k);
                mbar_expect_tx(&bar_ld[s], ST_TX + 256u);
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    tma_load_3d(st + ST_K + sl * T64, &mk, &bar_ld[s], 64 * sl, h, row0);
                    tma_load_3d(st + ST_Q + sl * T64, &mq, &bar_ld[s], 64 * sl, h, row0);
                    tma_load_3d(st + ST_O + sl * T64, &mo, &bar_ld[s], 64 * sl, h, row0);
                    tma_load_2d(st + ST_W + sl * T64, &mw, &bar_ld[s], 64 * sl, (int)(slot * C));
                }
                tma_load_2d(st + ST_A, &ma, &bar_ld[s], 0, (int)(slot * C));
                bulk_load(sg + s * 64, g_ws + slot * C, 256u, &bar_ld[s]);
            }
            __syncwarp();
        }
        if (sAbort)
            for (int r = k > NS ? k - NS : 0; r < k; ++r)
                (void)mbar_wait(&bar_ld[r % NS], (uint32_t)((r / NS) & 1));
    } else if (warp == NMAIN) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t id_x = idesc_bf16_f32(128, 64, false, false);   // dS'^T K^T
        constexpr uint32_t id_y = idesc_bf16_f32(128, 64, true, false);    // dO^T A_qk
        constexpr uint32_t id_q = idesc_bf16_f32(128, 128, true, true);    // dO^T (e^g Q)
        constexpr uint32_t id_w = idesc_bf16_f32(128, 128, false, true);   // (-dU^T) W
        const uint32_t aS = smem_u32(sS);
        // the chunk-input products of step k: Y, and the Q half of D into buffer k % 2
        auto issue_inputs = [&](int k) {
            const uint32_t st = smem_u32(sm + (k % NS) * ST_BYTES);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)   // A = dO (MN-major, M = j), B = A^T rows (K-major)
                mma_bf16(tb + TM_Y, sdesc_sw128(st + ST_O + ks * 2048, T64, 1024),
                         sdesc_sw128(st + ST_A + ks * 32, 16, 1024), id_y, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)   // B = e^g Q (MN-major, N = i)
                mma_bf16(tb + TM_D + 128u * (uint32_t)(k & 1),
                         sdesc_sw128(st + ST_O + ks * 2048, T64, 1024),
                         sdesc_sw128(st + ST_Q + ks * 2048, T64, 1024), id_q, ks > 0);
        };
        bool ok = true;
        if (nch > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bar_ld[0], 0u, &sAbort) &&
                                             mbar_wait_or_abort(&bar_prep, 0u, &sAbort));
            if (ok) {
                tc_fence_after();
                if (lane == 0) issue_inputs(0);
                __syncwarp();
            }
        }
        for (int k = 0; ok && k < nch; ++k) {
            const uint32_t st = smem_u32(sm + (k % NS) * ST_BYTES);
            // X = dS'^T K^T once dS'^T is in shared memory; dS' of the step's
            // chunk recorded as that bf16 tile (32 KB image)
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_s, (uint32_t)(k & 1), &sAbort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                bulk_store(dS_img + (size_t)slot_of(k) * 32768, sS, 32768u);
                bulk_commit_group();
            }
            if (lane == 0) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tb + TM_X, sdesc_sw128(aS + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                             sdesc_sw128(st + ST_K + (ks >> 2) * T64 + (ks & 3) * 32, 16, 1024),
                             id_x, ks > 0);
                mma_commit(&bar_x);
            }
            __syncwarp();
            // D += (-dU^T) W once dU^T (bf16) is in TMEM; the record has read
            // dS'^T before D lets the main warps overwrite it
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_u, (uint32_t)(k & 1), &sAbort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) bulk_wait_group_read0();
            if (lane == 0) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ts(tb + TM_D + 128u * (uint32_t)(k & 1), tb + TM_U + 8u * (uint32_t)ks,
                                sdesc_sw128(st + ST_W + ks * 2048, T64, 1024), id_w, 1);
                mma_commit(&bar_d);
                mma_commit(&bar_empty[k % NS]);
            }
            __syncwarp();
            // the next chunk's input products (Y is read, D buffer (k + 1) % 2 too)
            if (k + 1 < nch) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait_or_abort(&bar_ld[(k + 1) % NS], (uint32_t)(((k + 1) / NS) & 1),
                                                   &sAbort) &&
                                    mbar_wait_or_abort(&bar_prep, (uint32_t)((k + 1) & 1), &sAbort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) issue_inputs(k + 1);
                __syncwarp();
            }
        }
        if (!ok) fail();
        if (lane == 0) {
            mma_commit(&bar_fin);
            bulk_wait_group0();
        }
        __syncwarp();
        (void)mbar_wait(&bar_fin, 0u);
    } else {
        // ------------------------------------------------------------ main warps
        const int j = (warp & 3) * 32 + lane;   // column of dS (TMEM lane)
        const int hf = warp >> 2;               // rows i in [64 hf, 64 hf + 64)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        unsigned char *const sSrow = sS + hf * 16384;
        float ds[64];   // dS'^T[j][64 hf + x]
#pragma unroll
        for (int x = 0; x < 64; ++x)
            ds[x] = p.dS_T ? p.dS_T[sbase + (size_t)(64 * hf + x) * D + j] : 0.f;
        // bf16 row j of dS'^T into shared memory (the A operand of X)
        auto put_state = [&]() {
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(sSrow + sw128_offset(j, 8 * c8)) =
                    make_uint4(dtc_pack(ds[8 * c8], ds[8 * c8 + 1]), dtc_pack(ds[8 * c8 + 2], ds[8 * c8 + 3]),
                               dtc_pack(ds[8 * c8 + 4], ds[8 * c8 + 5]), dtc_pack(ds[8 * c8 + 6], ds[8 * c8 + 7]));
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_s);
        };
        // stage of step k landed: the rows past the sequence's end cleared (K,
        // Q, dO, A^T), Q scaled by exp g, the decay factors of the chunk
        const int mt = tid;   // 0 .. 255
        auto prep = [&](int k) -> bool {
            const int s = k % NS;
            if (!__all_sync(0xffffffffu,
                            mbar_wait_or_abort(&bar_ld[s], (uint32_t)((k / NS) & 1), &sAbort)))
                return false;
            unsigned char *st = sm + s * ST_BYTES;
            const int c = nch - 1 - k;
            const int nc = min(C, geo.len - c * C);
            const float *g = sg + s * 64;
            // thread: token t = mt >> 2, 16-byte pieces (mt & 3) + 4 u of its 16
            const int t = mt >> 2;
            const float et = __expf(g[t]);
            const bool live = t < nc;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int pc = (mt & 3) + 4 * u, sl = pc >> 3;
                const uint32_t off = sl * T64 + sw128_offset(t, 8 * (pc & 7));
                uint4 *q4 = reinterpret_cast<uint4 *>(st + ST_Q + off);
                uint4 w = *q4;
                if (live) {
                    w = make_uint4(dtc_pack(et * __uint_as_float(w.x << 16), et * __uint_as_float(w.x & 0xffff0000u)),
                                   dtc_pack(et * __uint_as_float(w.y << 16), et * __uint_as_float(w.y & 0xffff0000u)),
                                   dtc_pack(et * __uint_as_float(w.z << 16), et * __uint_as_float(w.z & 0xffff0000u)),
                                   dtc_pack(et * __uint_as_float(w.w << 16), et * __uint_as_float(w.w & 0xffff0000u)));
                } else {
                    w = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(st + ST_K + off) = w;
                    *reinterpret_cast<uint4 *>(st + ST_O + off) = w;
                    if (u < 2)   // A^T row t: 8 pieces
                        *reinterpret_cast<uint4 *>(st + ST_A + sw128_offset(t, 8 * ((mt & 3) + 4 * u))) = w;
                }
                *q4 = w;
            }
            if (mt < 64) {
                se[s * 128 + mt] = __expf(g[mt]);
                se[s * 128 + 64 + mt] = __expf(g[C - 1] - g[mt]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_prep);
            return true;
        };

        bool ok = true;
        if (nch > 0) {
            put_state();
            ok = prep(0);
            if (!ok) fail();
        }
        for (int k = 0; ok && k < nch; ++k) {
            const int s = k % NS;
            // ---- dU^T = X diag(exp(g_C - g)) + Y for tokens t in [32 hf, 32 hf + 32)
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_x, (uint32_t)(k & 1), &sAbort))) {
                fail();
                break;
            }
            tc_fence_after();
            {
                uint32_t xr[32], yr[32];
                tmem_ld32(tb + lane_base + TM_X + 32 * hf, xr);
                tmem_ld32(tb + lane_base + TM_Y + 32 * hf, yr);
                tmem_ld_wait();
                const float *egc = se + s * 128 + 64 + 32 * hf;
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float u0 = fmaf(egc[2 * e], __uint_as_float(xr[2 * e]), __uint_as_float(yr[2 * e]));
                    const float u1 = fmaf(egc[2 * e + 1], __uint_as_float(xr[2 * e + 1]),
                                          __uint_as_float(yr[2 * e + 1]));
                    w[e] = dtc_pack(-u0, -u1);
                }
                tmem_st16(tb + lane_base + TM_U + 16 * hf, w);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_u);
            // ---- the next chunk's stage, while D is completed
            if (k + 1 < nch && !prep(k + 1)) {
                fail();
                break;
            }
            // ---- dS'^T <- exp(g_C) dS'^T + D
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_d, (uint32_t)(k & 1), &sAbort))) {
                fail();
                break;
            }
            tc_fence_after();
            {
                const float egC = se[s * 128 + C - 1];   // exp(g_C)
                const uint32_t tD = tb + lane_base + TM_D + 128u * (uint32_t)(k & 1) + 64u * hf;
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t r[32];
                    tmem_ld32(tD + 32 * c2, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        ds[32 * c2 + x] = fmaf(egC, ds[32 * c2 + x], __uint_as_float(r[x]));
                }
            }
            tc_fence_before();
            if (k + 1 < nch) put_state();
        }
        if (ok && !sAbort && p.dS0) {
#pragma unroll
            for (int x = 0; x < 64; ++x) p.dS0[sbase + (size_t)(64 * hf + x) * D + j] = ds[x];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// ------------------------------------------------------------ token gradients
// Row strides are multiples of 4 floats so that the products read float4
// operands; every product runs on 2D register tiles:
//   layout A (64 x D outputs): tokens 2 tp, 2 tp + 1 x columns cg JT .. + JT;
//   layout B (64 x 64 outputs): tokens 4 tb + m x positions sb + 16 n;
//   layout P (products with rows of S or dS'): tokens 2 tp, 2 tp + 1 x rows
//   cg + 8 n.
// The rows a thread reads in layouts B and P are 16 or 8 apart, so that the
// float4 loads of a warp spread over all banks.
template <int D>
struct GrSmem {
    static constexpr int LK = D + 4, LM = C + 4;
    float K[C][LK], Q[C][LK];
    float M0[C][LM];   // raw strict-lower K K^T, its dg terms, then X + X^T
    float M1[C][LM];   // raw lower Q K^T, its dg terms, then dA_qk o Gamma
    float M2[C][LM];   // T, then X = diag(beta) (dA_kk o Gamma)
    float tA[C][LK];   // A_kk and S / dS' rows (staging), then U
    float tB[C][LK];   // V - diag(exp g) K S, then dR
    float tC[C][LK];   // dO, then dU, then S and dS' row blocks (staging)
    Vec v;
    float dbeta[C], dg[C], dgcol[C], red[NT / 32];
    float scr[32 * 33];   // scratch of the triangular inverse
};

// Column sums of the [C][LM] matrix E over rows r >= s (threads 0..63).
template <int LM>
__device__ __forceinline__ void col_sums(const float (*E)[LM], float *dgcol, int tid) {
    if (tid < C) {
        float sg = 0.f;
        for (int r = tid; r < C; ++r) sg += E[r][tid];
        dgcol[tid] = sg;
    }
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// N consecutive input values (N a multiple of 4) as floats.
template <int N>
__device__ __forceinline__ void ld_row(const float *p, float (&f)[N]) {
#pragma unroll
    for (int k = 0; k < N / 4; ++k) {
        const float4 v = *reinterpret_cast<const float4 *>(p + 4 * k);
        f[4 * k] = v.x; f[4 * k + 1] = v.y; f[4 * k + 2] = v.z; f[4 * k + 3] = v.w;
    }
}
template <int N>
__device__ __forceinline__ void ld_row(const __nv_bfloat16 *p, float (&f)[N]) {
#pragma unroll
    for (int k = 0; k < N / 4; ++k) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p + 4 * k);
        f[4 * k] = __uint_as_float(v.x << 16); f[4 * k + 1] = __uint_as_float(v.x & 0xffff0000u);
        f[4 * k + 2] = __uint_as_float(v.y << 16); f[4 * k + 3] = __uint_as_float(v.y & 0xffff0000u);
    }
}
template <int N>
__device__ __forceinline__ void st_row(float *p, const float (&f)[N]) {
#pragma unroll
    for (int k = 0; k < N / 4; ++k)
        *reinterpret_cast<float4 *>(p + 4 * k) = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
}
template <int N>
__device__ __forceinline__ void st_row(__nv_bfloat16 *p, const float (&f)[N]) {
#pragma unroll
    for (int k = 0; k < N / 4; ++k) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(f[4 * k], f[4 * k + 1]);
        const __nv_bfloat162 c = __floats2bfloat162_rn(f[4 * k + 2], f[4 * k + 3]);
        *reinterpret_cast<uint2 *>(p + 4 * k) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&c));
    }
}

// Raw Gram products for rows of stride LK (a multiple of 4): Mkk = strict
// lower K K^T, Mqk = lower Q K^T.  Thread (bt, bs) forms rows bt + 16 m x
// columns bs + 16 n of both, reading float4 along the features: the 16 rows
// a warp reads per load are 16 apart (two wavefronts, the minimum for 16
// distinct float4 rows).
template <int D, int LK, int LM>
__device__ void gram_v(const float (*K)[LK], const float (*Q)[LK], float (*Mkk)[LM],
                       float (*Mqk)[LM], int tid) {
    const int bt = tid >> 4, bs = tid & 15;
    float akk[4][4], aqk[4][4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) akk[m][n] = aqk[m][n] = 0.f;
#pragma unroll 2
    for (int i = 0; i < D; i += 4) {
        float4 kt[4], qt[4], ks[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            kt[m] = ld4(&K[bt + 16 * m][i]);
            qt[m] = ld4(&Q[bt + 16 * m][i]);
            ks[m] = ld4(&K[bs + 16 * m][i]);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                akk[m][n] += dot4(kt[m], ks[n]);
                aqk[m][n] += dot4(qt[m], ks[n]);
            }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int t = bt + 16 * m, s2 = bs + 16 * n;
            Mkk[t][s2] = s2 < t ? akk[m][n] : 0.f;
            Mqk[t][s2] = s2 <= t ? aqk[m][n] : 0.f;
        }
}

template <typename Tin, int D>
__global__ void __launch_bounds__(NT, 1) bwd_grads_kernel(BwdProblem p, int nch_fixed,
                                                          const float *S_chk,
                                                          const float *dS_chk) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    using Sm = GrSmem<D>;
    constexpr int LK = Sm::LK, LM = Sm::LM;
    constexpr int JT = D / 8;   // layout A: columns per thread
    constexpr int IB = 32;      // rows of S and dS' per staged block
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);
    const int tid = threadIdx.x;
    // one CTA per chunk slot: global chunk blockIdx.x, head blockIdx.y
    const long gch = blockIdx.x;
    const int h = blockIdx.y;
    if (p.status != nullptr && *(volatile unsigned *)p.status != kDevOk) return;
    if (p.cu_seqlens && gch >= p.chunk_prefix[p.n_seq]) return;   // past the last chunk
    const int seq = p.cu_seqlens ? p.chunk_seq[gch] : (int)(gch / nch_fixed);
    const SeqGeo sq = seq_geo(p, seq);
    const int c = (int)(gch - sq.chunk0);
    const long row0 = sq.start + (long)c * C;
    const int nc = min(C, sq.len - c * C);
    const size_t slot = (size_t)gch * p.H + h;
    const float *S = S_chk + slot * D * D;     // state at the chunk start
    const float *dSp = dS_chk + slot * D * D;  // gradient at its end
    const Tin *dout = static_cast<const Tin *>(p.dout);
    const Tin *vin = static_cast<const Tin *>(p.v);
    // layout A / P thread coordinates
    const int tp = tid >> 3, cg = tid & 7;
    const int ta[2] = {2 * tp, 2 * tp + 1};
    // layout A columns of this thread: 4 cg + 32 q + e (q < JT / 4, e < 4)
    auto colA = [cg](int q) { return 4 * cg + 32 * q; };
    const bool liveA[2] = {ta[0] < nc, ta[1] < nc};
    const size_t rowA[2] = {(size_t)(row0 + (liveA[0] ? ta[0] : 0)) * p.H + h,
                            (size_t)(row0 + (liveA[1] ? ta[1] : 0)) * p.H + h};
    // layout B
    const int tb = tid >> 4, sb = tid & 15;

    load_tile<Tin, C, D, LK, NT>(&sm.K[0][0], static_cast<const Tin *>(p.k), row0, nc, p.H, h, D,
                                 0, tid);
    load_tile<Tin, C, D, LK, NT>(&sm.Q[0][0], static_cast<const Tin *>(p.q), row0, nc, p.H, h, D,
                                 0, tid);
    load_tile<Tin, C, D, LK, NT>(&sm.tC[0][0], dout, row0, nc, p.H, h, D, 0, tid);
    if (tid < C) {
        const bool ok = tid < nc;
        const size_t r = (size_t)(row0 + tid) * p.H + h;
        sm.v.alpha[tid] = (ok && p.alpha) ? p.alpha[r] : 1.f;
        sm.v.eta[tid] = ok ? p.eta[r] : 0.f;
    }
    __syncthreads();
    chunk_vectors<D, LK>(sm.K, sm.v, p.eps, p.beta_mode, nc, tid);
    __syncthreads();
    gram_v<D, LK, LM>(sm.K, sm.Q, sm.M0, sm.M1, tid);
    __syncthreads();
    {   // A_kk = strict_lower(beta Gamma o K K^T) into tA, then T
        float(*Akk)[LM] = reinterpret_cast<float(*)[LM]>(&sm.tA[0][0]);
        for (int x = tid; x < C * C; x += NT) {
            const int r = x / C, s2 = x % C;
            Akk[r][s2] = s2 < r ? sm.v.beta[r] * gam(sm.v, r, s2) * sm.M0[r][s2] : 0.f;
        }
        __syncthreads();
        invert_unit_lower64<LM, LM>(Akk, sm.M2, sm.scr, tid);
    }
    // dO S^T for rows i = cg + 8 n of S (layout P), formed while S is staged
    float pq[2][D / 8];
    {   // (A) V - diag(exp g) K S -> tB, S staged in tA 64 rows at a time
        float acc[2][JT], vv[2][JT];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int q = 0; q < JT / 4; ++q) {
                float v4[4];
                ld_row<4>(vin + rowA[m] * D + colA(q), v4);
#pragma unroll
                for (int e = 0; e < 4; ++e) vv[m][4 * q + e] = liveA[m] ? v4[e] : 0.f;
            }
#pragma unroll
            for (int x = 0; x < JT; ++x) acc[m][x] = 0.f;
        }
#pragma unroll
        for (int i0 = 0; i0 < D; i0 += C) {
            load_block_f32<C, D, LK, NT>(&sm.tA[0][0], S + (size_t)i0 * D, D, tid);
            __syncthreads();
#pragma unroll 2
            for (int i = 0; i < C; ++i) {
                const float k0 = sm.K[ta[0]][i0 + i], k1 = sm.K[ta[1]][i0 + i];
#pragma unroll
                for (int q = 0; q < JT / 4; ++q) {
                    const float4 s4 = ld4(&sm.tA[i][colA(q)]);
                    acc[0][4 * q] = fmaf(k0, s4.x, acc[0][4 * q]); acc[0][4 * q + 1] = fmaf(k0, s4.y, acc[0][4 * q + 1]);
                    acc[0][4 * q + 2] = fmaf(k0, s4.z, acc[0][4 * q + 2]); acc[0][4 * q + 3] = fmaf(k0, s4.w, acc[0][4 * q + 3]);
                    acc[1][4 * q] = fmaf(k1, s4.x, acc[1][4 * q]); acc[1][4 * q + 1] = fmaf(k1, s4.y, acc[1][4 * q + 1]);
                    acc[1][4 * q + 2] = fmaf(k1, s4.z, acc[1][4 * q + 2]); acc[1][4 * q + 3] = fmaf(k1, s4.w, acc[1][4 * q + 3]);
                }
            }
            // pq[t][i0 + cg + 8 n] = dO_t . S_i for the 8 staged rows of this thread
            float pp[2][8];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 8; ++n) pp[m][n] = 0.f;
#pragma unroll 2
            for (int j = 0; j < D; j += 4) {
                const float4 o0 = ld4(&sm.tC[ta[0]][j]), o1 = ld4(&sm.tC[ta[1]][j]);
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    const float4 s4 = ld4(&sm.tA[cg + 8 * n][j]);
                    pp[0][n] += dot4(o0, s4);
                    pp[1][n] += dot4(o1, s4);
                }
            }
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 8; ++n) pq[m][i0 / 8 + n] = pp[m][n];
            __syncthreads();
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const float e = sm.v.eg[ta[m]];
#pragma unroll
            for (int x = 0; x < JT; ++x) acc[m][x] = vv[m][x] - e * acc[m][x];
#pragma unroll
            for (int q = 0; q < JT / 4; ++q)
                *reinterpret_cast<float4 *>(&sm.tB[ta[m]][colA(q)]) =
                    make_float4(acc[m][4 * q], acc[m][4 * q + 1], acc[m][4 * q + 2], acc[m][4 * q + 3]);
        }
    }
    __syncthreads();
    float du[2][JT];
    {   // (A) U = T diag(beta) (V - e^g K S);  dU = A_qk^T dO + diag(exp(g_C - g)) K dS'
        float u[2][JT];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int x = 0; x < JT; ++x) u[m][x] = du[m][x] = 0.f;
        for (int s2 = 0; s2 <= ta[1]; ++s2) {   // T is lower triangular
            const float bs = sm.v.beta[s2];
            const float a0 = sm.M2[ta[0]][s2] * bs, a1 = sm.M2[ta[1]][s2] * bs;
#pragma unroll
            for (int q = 0; q < JT / 4; ++q) {
                const float4 w = ld4(&sm.tB[s2][colA(q)]);
                u[0][4 * q] = fmaf(a0, w.x, u[0][4 * q]); u[0][4 * q + 1] = fmaf(a0, w.y, u[0][4 * q + 1]);
                u[0][4 * q + 2] = fmaf(a0, w.z, u[0][4 * q + 2]); u[0][4 * q + 3] = fmaf(a0, w.w, u[0][4 * q + 3]);
                u[1][4 * q] = fmaf(a1, w.x, u[1][4 * q]); u[1][4 * q + 1] = fmaf(a1, w.y, u[1][4 * q + 1]);
                u[1][4 * q + 2] = fmaf(a1, w.z, u[1][4 * q + 2]); u[1][4 * q + 3] = fmaf(a1, w.w, u[1][4 * q + 3]);
            }
        }
        for (int s2 = ta[0]; s2 < C; ++s2) {   // A_qk[s][t] = Gamma_st (q_s . k_t), s >= t
            const float a0 = gam(sm.v, s2, ta[0]) * sm.M1[s2][ta[0]];
            const float a1 = s2 >= ta[1] ? gam(sm.v, s2, ta[1]) * sm.M1[s2][ta[1]] : 0.f;
#pragma unroll
            for (int q = 0; q < JT / 4; ++q) {
                const float4 o = ld4(&sm.tC[s2][colA(q)]);
                du[0][4 * q] = fmaf(a0, o.x, du[0][4 * q]); du[0][4 * q + 1] = fmaf(a0, o.y, du[0][4 * q + 1]);
                du[0][4 * q + 2] = fmaf(a0, o.z, du[0][4 * q + 2]); du[0][4 * q + 3] = fmaf(a0, o.w, du[0][4 * q + 3]);
                du[1][4 * q] = fmaf(a1, o.x, du[1][4 * q]); du[1][4 * q + 1] = fmaf(a1, o.y, du[1][4 * q + 1]);
                du[1][4 * q + 2] = fmaf(a1, o.z, du[1][4 * q + 2]); du[1][4 * q + 3] = fmaf(a1, o.w, du[1][4 * q + 3]);
            }
        }
        const float e0 = sm.v.egc[ta[0]], e1 = sm.v.egc[ta[1]];
        for (int i0 = 0; i0 < D; i0 += C) {
            load_block_f32<C, D, LK, NT>(&sm.tA[0][0], dSp + (size_t)i0 * D, D, tid);
            __syncthreads();
#pragma unroll 2
            for (int i = 0; i < C; ++i) {
                const float k0 = e0 * sm.K[ta[0]][i0 + i], k1 = e1 * sm.K[ta[1]][i0 + i];
#pragma unroll
                for (int q = 0; q < JT / 4; ++q) {
                    const float4 d4 = ld4(&sm.tA[i][colA(q)]);
                    du[0][4 * q] = fmaf(k0, d4.x, du[0][4 * q]); du[0][4 * q + 1] = fmaf(k0, d4.y, du[0][4 * q + 1]);
                    du[0][4 * q + 2] = fmaf(k0, d4.z, du[0][4 * q + 2]); du[0][4 * q + 3] = fmaf(k0, d4.w, du[0][4 * q + 3]);
                    du[1][4 * q] = fmaf(k1, d4.x, du[1][4 * q]); du[1][4 * q + 1] = fmaf(k1, d4.y, du[1][4 * q + 1]);
                    du[1][4 * q + 2] = fmaf(k1, d4.z, du[1][4 * q + 2]); du[1][4 * q + 3] = fmaf(k1, d4.w, du[1][4 * q + 3]);
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < JT / 4; ++q)
                *reinterpret_cast<float4 *>(&sm.tA[ta[m]][colA(q)]) =
                    make_float4(u[m][4 * q], u[m][4 * q + 1], u[m][4 * q + 2], u[m][4 * q + 3]);
    }
    __syncthreads();
    {   // (B) dA_qk = lower(dO U^T); its Gamma terms of dg; M1 <- dA_qk o Gamma
        float da[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) da[m][n] = 0.f;
#pragma unroll 2
        for (int j = 0; j < D; j += 4) {
            float4 o[4], u4[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) o[m] = ld4(&sm.tC[4 * tb + m][j]);
#pragma unroll
            for (int n = 0; n < 4; ++n) u4[n] = ld4(&sm.tA[sb + 16 * n][j]);
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n) da[m][n] += dot4(o[m], u4[n]);
        }
        float rs[4], ev[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            rs[m] = 0.f;
            const int t = 4 * tb + m;
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int s2 = sb + 16 * n;
                const float ga = s2 <= t ? gam(sm.v, t, s2) : 0.f;
                da[m][n] = s2 <= t ? da[m][n] * ga : 0.f;   // dA_qk o Gamma
                ev[m][n] = da[m][n] * sm.M1[t][s2];         // dA_qk o A_qk
                rs[m] += ev[m][n];
            }
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) rs[m] += __shfl_xor_sync(0xffffffffu, rs[m], off);
        }
        __syncthreads();   // dO reads and raw Q K^T reads are complete
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) sm.M1[4 * tb + m][sb + 16 * n] = ev[m][n];
        __syncthreads();
        col_sums<LM>(sm.M1, sm.dgcol, tid);
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) sm.M1[4 * tb + m][sb + 16 * n] = da[m][n];
#pragma unroll
        for (int m = 0; m < 2; ++m)   // dU
#pragma unroll
            for (int q = 0; q < JT / 4; ++q)
                *reinterpret_cast<float4 *>(&sm.tC[ta[m]][colA(q)]) =
                    make_float4(du[m][4 * q], du[m][4 * q + 1], du[m][4 * q + 2], du[m][4 * q + 3]);
        if (sb == 0) {
#pragma unroll
            for (int m = 0; m < 4; ++m) sm.dg[4 * tb + m] = rs[m] - sm.dgcol[4 * tb + m];
        }
    }
    __syncthreads();
    {   // (A) dR = T^T dU; dbeta and dg from R = diag(beta)(V - e^g K S); dV
        float dr[2][JT];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int x = 0; x < JT; ++x) dr[m][x] = 0.f;
        for (int s2 = ta[0]; s2 < C; ++s2) {   // T[s][t], s >= t
            const float a0 = sm.M2[s2][ta[0]], a1 = sm.M2[s2][ta[1]];
#pragma unroll
            for (int q = 0; q < JT / 4; ++q) {
                const float4 w = ld4(&sm.tC[s2][colA(q)]);
                dr[0][4 * q] = fmaf(a0, w.x, dr[0][4 * q]); dr[0][4 * q + 1] = fmaf(a0, w.y, dr[0][4 * q + 1]);
                dr[0][4 * q + 2] = fmaf(a0, w.z, dr[0][4 * q + 2]); dr[0][4 * q + 3] = fmaf(a0, w.w, dr[0][4 * q + 3]);
                dr[1][4 * q] = fmaf(a1, w.x, dr[1][4 * q]); dr[1][4 * q + 1] = fmaf(a1, w.y, dr[1][4 * q + 1]);
                dr[1][4 * q + 2] = fmaf(a1, w.z, dr[1][4 * q + 2]); dr[1][4 * q + 3] = fmaf(a1, w.w, dr[1][4 * q + 3]);
            }
        }
        float p1[2] = {0.f, 0.f}, p2[2] = {0.f, 0.f};
        Tin *dvo = static_cast<Tin *>(p.dv);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const float bt = sm.v.beta[ta[m]];
#pragma unroll
            for (int q = 0; q < JT / 4; ++q) {
                float vv[4], dvv[4];
                ld_row<4>(vin + rowA[m] * D + colA(q), vv);
                const float4 w4 = ld4(&sm.tB[ta[m]][colA(q)]);
                const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float d = dr[m][4 * q + e];
                    p1[m] = fmaf(wv[e], d, p1[m]);
                    p2[m] = fmaf(liveA[m] ? vv[e] : 0.f, d, p2[m]);
                    dvv[e] = bt * d;
                }
                if (liveA[m]) st_row<4>(dvo + rowA[m] * D + colA(q), dvv);
            }
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                p1[m] += __shfl_xor_sync(0xffffffffu, p1[m], off);
                p2[m] += __shfl_xor_sync(0xffffffffu, p2[m], off);
            }
        }
        __syncthreads();   // V - e^g K S, dU and T fully read
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < JT / 4; ++q)
                *reinterpret_cast<float4 *>(&sm.tB[ta[m]][colA(q)]) =
                    make_float4(dr[m][4 * q], dr[m][4 * q + 1], dr[m][4 * q + 2], dr[m][4 * q + 3]);
        if (cg == 0) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                sm.dbeta[ta[m]] = p1[m];
                sm.dg[ta[m]] += sm.v.beta[ta[m]] * (p1[m] - p2[m]);   // -beta e^g (K S)_t . dR_t
            }
        }
    }
    __syncthreads();
    {   // (B) dA_kk = -strict_lower(dR U^T); its terms of dg and dbeta; M2 <- X
        float dk2[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) dk2[m][n] = 0.f;
#pragma unroll 2
        for (int j = 0; j < D; j += 4) {
            float4 r4[4], u4[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) r4[m] = ld4(&sm.tB[4 * tb + m][j]);
#pragma unroll
            for (int n = 0; n < 4; ++n) u4[n] = ld4(&sm.tA[sb + 16 * n][j]);
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n) dk2[m][n] += dot4(r4[m], u4[n]);
        }
        float rs[4], rb[4], fv[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int t = 4 * tb + m;
            const float bt = sm.v.beta[t];
            rs[m] = rb[m] = 0.f;
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int s2 = sb + 16 * n;
                const float xg = s2 < t ? -dk2[m][n] * gam(sm.v, t, s2) : 0.f;   // dA_kk o Gamma
                const float e = xg * sm.M0[t][s2];                               // . K K^T
                rb[m] += e;
                rs[m] += bt * e;                                                 // dA_kk o A_kk
                fv[m][n] = bt * e;
                dk2[m][n] = bt * xg;                                             // X
            }
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) {
                rs[m] += __shfl_xor_sync(0xffffffffu, rs[m], off);
                rb[m] += __shfl_xor_sync(0xffffffffu, rb[m], off);
            }
        }
        __syncthreads();   // raw K K^T reads complete
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                sm.M0[4 * tb + m][sb + 16 * n] = fv[m][n];
                sm.M2[4 * tb + m][sb + 16 * n] = dk2[m][n];
            }
        if (sb == 0) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                sm.dg[4 * tb + m] += rs[m];
                sm.dbeta[4 * tb + m] += rb[m];
            }
        }
        __syncthreads();
        col_sums<LM>(sm.M0, sm.dgcol, tid);
        __syncthreads();
        if (tid < C) sm.dg[tid] -= sm.dgcol[tid];
#pragma unroll
        for (int m = 0; m < 4; ++m)   // M0 <- X + X^T
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int t = 4 * tb + m, s2 = sb + 16 * n;
                sm.M0[t][s2] = sm.M2[t][s2] + sm.M2[s2][t];
            }
    }
    __syncthreads();
    // (P) dQ and dK; S and dS' staged in tC 32 rows at a time
    float(*Sb)[LK] = reinterpret_cast<float(*)[LK]>(&sm.tC[0][0]);
    float(*Db)[LK] = Sb + IB;
    float eg[2], egc[2], bt[2], cn[2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int t = ta[m];
        eg[m] = sm.v.eg[t]; egc[m] = sm.v.egc[t]; bt[m] = sm.v.beta[t];
        cn[m] = 0.f;   // the gradient through beta's key norm
        if (p.beta_mode == 0 && sm.v.den[t] != 0.f) {
            const float den = sm.v.den[t];
            cn[m] = -2.f * sm.v.eta[t] * sm.dbeta[t] / (den * den);
        }
    }
    float gq[2] = {0.f, 0.f}, gk[2] = {0.f, 0.f}, sds = 0.f;
    Tin *dqo = static_cast<Tin *>(p.dq);
    Tin *dko = static_cast<Tin *>(p.dk);
#pragma unroll
    for (int i0 = 0; i0 < D; i0 += IB) {
        __syncthreads();   // the previous block is fully read
        load_block_f32<IB, D, LK, NT>(&Sb[0][0], S + (size_t)i0 * D, D, tid);
        load_block_f32<IB, D, LK, NT>(&Db[0][0], dSp + (size_t)i0 * D, D, tid);
        __syncthreads();
        for (int x = tid; x < IB * D; x += NT) sds = fmaf(Sb[x / D][x % D], Db[x / D][x % D], sds);
        float pr[2][4], pu[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) pr[m][n] = pu[m][n] = 0.f;
#pragma unroll 2
        for (int j = 0; j < D; j += 4) {
            float4 r4[2], u4[2], s4[4], d4[4];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                r4[m] = ld4(&sm.tB[ta[m]][j]);
                u4[m] = ld4(&sm.tA[ta[m]][j]);
            }
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                s4[n] = ld4(&Sb[cg + 8 * n][j]);
                d4[n] = ld4(&Db[cg + 8 * n][j]);
            }
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    pr[m][n] += dot4(r4[m], s4[n]);
                    pu[m][n] += dot4(u4[m], d4[n]);
                }
        }
        // (dA_qk o Gamma) K, its transpose times Q, (X + X^T) K
        float dq[2][4], dkk[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) dq[m][n] = dkk[m][n] = 0.f;
#pragma unroll 2
        for (int s2 = 0; s2 < C; ++s2) {
            float kv[4], qv[4];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                kv[n] = sm.K[s2][i0 + cg + 8 * n];
                qv[n] = sm.Q[s2][i0 + cg + 8 * n];
            }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const float a_ts = sm.M1[ta[m]][s2], a_st = sm.M1[s2][ta[m]], x2 = sm.M0[ta[m]][s2];
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    dq[m][n] = fmaf(a_ts, kv[n], dq[m][n]);
                    dkk[m][n] = fmaf(a_st, qv[n], fmaf(x2, kv[n], dkk[m][n]));
                }
            }
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int i = i0 + cg + 8 * n;
                const float kv = sm.K[ta[m]][i], qv = sm.Q[ta[m]][i];
                const float pqv = pq[m][i0 / 8 + n];
                dq[m][n] = fmaf(eg[m], pqv, dq[m][n]);
                dkk[m][n] = fmaf(-bt[m] * eg[m], pr[m][n], dkk[m][n]);
                dkk[m][n] = fmaf(egc[m], pu[m][n], dkk[m][n]);
                dkk[m][n] = fmaf(cn[m], kv, dkk[m][n]);
                gq[m] = fmaf(qv, pqv, gq[m]);
                gk[m] = fmaf(kv, pu[m][n], gk[m]);
                if (liveA[m]) {
                    dqo[rowA[m] * D + i] = static_cast<Tin>(dq[m][n]);
                    dko[rowA[m] * D + i] = static_cast<Tin>(dkk[m][n]);
                }
            }
        }
    }
    // dg: exp(g) of the Q S read, exp(g_C - g) of the state write; dg_C: the
    // state write and exp(g_C) S
    float red = sm.v.eg[C - 1] * sds;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) {
            gq[m] += __shfl_xor_sync(0xffffffffu, gq[m], off);
            gk[m] += __shfl_xor_sync(0xffffffffu, gk[m], off);
        }
        const float wk = egc[m] * gk[m];
        if (cg == 0) {
            sm.dg[ta[m]] += eg[m] * gq[m] - wk;
            red += wk;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) red += __shfl_xor_sync(0xffffffffu, red, off);
    if ((tid & 31) == 0) sm.red[tid >> 5] = red;
    __syncthreads();
    if (tid < 32) {   // dg_C onto g_{C-1}; reverse cumulative sum -> dlog(alpha)
        float gc = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) gc += sm.red[w];
        const int lane = tid;
        float d0 = sm.dg[lane], d1 = sm.dg[lane + 32];
        if (lane == 31) d1 += gc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {   // suffix sums
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
                    const float dbt = sm.dbeta[tt];
                    const float den = sm.v.den[tt];
                    p.deta[r] = p.beta_mode ? dbt : (den != 0.f ? dbt / den : 0.f);
                }
            }
        }
    }
}

// ------------------------------------------------------ token gradients (tcgen05)
// bf16 with d = 128: per chunk, the products of the gradient lines above on
// the tensor cores, from the recorded S and dS'^T (bf16 operand tiles as the
// forward's state pass and the dS chain held them, loaded by bulk copies),
// the forward's T (bf16) and A^T, g of the chunk workspace.
// Every product has M = 128 token rows: a chunk has 64, so two 64-row tiles
// stored slab by slab one after the other act as one 128-row operand and
// share the product ([dR ; dO] S^T gives dR S^T and dO S^T = pq; [dR ; dO] U^T
// gives dR U^T and dO U^T; [X + X^T ; M1] K with M1 = dA_qk o Gamma); where
// only one tile is meant, the other 64 rows are whatever follows it in shared
// memory and their accumulator lanes are not read.  TMEM lane t holds token
// t's row (lanes 64 + t: the second tile's token t).  Four product phases,
// each followed by its epilogue on the CUDA cores:
//   1. K S, A_qk^T dO, K dS', K K^T (lanes 64..: Q K^T)
//      -> R = diag(beta)(V - diag(exp g) K S), dU = A_qk^T dO + diag(exp(g_C - g)) K dS'
//   2. U = T R, dR = T^T dU  -> dV = diag(beta) dR, dbeta and dg from R
//   3. [dR ; dO] U^T, U dS'^T, [dR ; dO] S^T  -> M1, X, their dg and dbeta terms
//   4. [X + X^T ; M1] K + M1^T Q  -> dQ (lanes 64..), dK (lanes 0..63)
// Shared memory (offsets in KB): [K | Q] 0, [dR | dO] 32, V 64, S 80, dS'^T 112,
// T 144, A^T 152, R 160, U 176, dU 192, vectors 208; reused: dV staging and
// then [X + X^T | M1] in R, the column-sum scratch in dS'^T, T and A^T, X
// (fp32) in S, zeros in U, dK staging in S and dQ staging in dU.
namespace gtc {
constexpr uint32_t KB = 1024;
constexpr uint32_t SL = 8 * KB;        // one 64 x 64 bf16 slab (64 rows of 128 bytes)
constexpr uint32_t O_KQ = 0, O_RO = 32 * KB, O_V = 64 * KB, O_S = 80 * KB, O_DS = 112 * KB,
                   O_T = 144 * KB, O_A = 152 * KB, O_R = 160 * KB, O_U = 176 * KB,
                   O_DU = 192 * KB, O_VEC = 208 * KB;
constexpr uint32_t SMEM = O_VEC + 4 * KB + 1024;
constexpr int NTH = 256;               // 8 warps: 2 per TMEM lane quadrant
constexpr uint32_t C_A = 0, C_B = 128, C_C = 256, C_G = 384;   // TMEM columns
static_assert(SMEM <= 232448, "gradient kernel shared memory");
}  // namespace gtc

// A 128-row K-major operand over two 64-row tiles stored slab by slab, one
// slab pair every `pair` bytes (K step of 16 = 32 bytes within a slab).
__device__ __forceinline__ uint64_t gk_desc(uint32_t base, int ks, uint32_t pair) {
    return tc::sdesc_sw128(base + (uint32_t)(ks >> 2) * pair + (uint32_t)(ks & 3) * 32u, 16, 1024);
}
// An MN-major operand: K step of 16 rows = 2048 bytes, the 64-element MN
// halves `lbo` bytes apart.
__device__ __forceinline__ uint64_t gm_desc(uint32_t base, int ks, uint32_t lbo) {
    return tc::sdesc_sw128(base + (uint32_t)ks * 2048u, lbo, 1024);
}
__device__ __forceinline__ uint32_t g_pack(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ float g_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float g_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
// Element (row, col) of a 64-column bf16 slab with the 128-byte swizzle.
__device__ __forceinline__ float g_at(const unsigned char *slab, int row, int col) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(slab + tc::sw128_offset(row, col)));
}
// 16 fp32 values -> bf16 columns [c0, c0 + 16) of row `row` of a slab.
__device__ __forceinline__ void g_st16(unsigned char *slab, int row, int c0, const float *x) {
#pragma unroll
    for (int k = 0; k < 2; ++k)
        *reinterpret_cast<uint4 *>(slab + tc::sw128_offset(row, c0 + 8 * k)) =
            make_uint4(g_pack(x[8 * k], x[8 * k + 1]), g_pack(x[8 * k + 2], x[8 * k + 3]),
                       g_pack(x[8 * k + 4], x[8 * k + 5]), g_pack(x[8 * k + 6], x[8 * k + 7]));
}

__global__ void __launch_bounds__(gtc::NTH, 1)
bwd_grads_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
                    const __grid_constant__ CUtensorMap mt, const __grid_constant__ CUtensorMap ma,
                    const __grid_constant__ CUtensorMap mdq, const __grid_constant__ CUtensorMap mdk,
                    const __grid_constant__ CUtensorMap mdv, BwdProblem p, int nch_fixed,
                    const unsigned char *S_img, const unsigned char *dS_img, const float *g_ws) {
    using namespace gtc;
    using namespace tc;
    extern __shared__ unsigned char g_smem[];
    unsigned char *sm = g_smem + ((1024u - (smem_u32(g_smem) & 1023u)) & 1023u);
    __shared__ uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tslot;
    __shared__ int sBad;
    float *vec = reinterpret_cast<float *>(sm + O_VEC);
    float *vg = vec, *veg = vec + 64, *vegc = vec + 128, *vbeta = vec + 192, *vden = vec + 256,
          *veta = vec + 320, *valpha = vec + 384, *vdbeta = vec + 448, *vdg = vec + 512,
          *vp = vec + 576 /* [2][2][64]: the halves' p1, p2 */, *vred = vec + 832 /* [8] */;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long gch = blockIdx.x;
    const int h = blockIdx.y;
    if (p.status != nullptr && *(volatile unsigned *)p.status != kDevOk) return;
    if (p.cu_seqlens && gch >= p.chunk_prefix[p.n_seq]) return;   // past the last chunk
    const int seq = p.cu_seqlens ? p.chunk_seq[gch] : (int)(gch / nch_fixed);
    const SeqGeo sq = seq_geo(p, seq);
    const int c = (int)(gch - sq.chunk0);
    const long row0 = sq.start + (long)c * C;
    const int nc = min(C, sq.len - c * C);
    const size_t slot = (size_t)gch * p.H + h;
    // TMEM lane of this thread and its column half; rows 0..63 live in warps
    // 0, 1, 4, 5 (lower), the second tile's rows in warps 2, 3, 6, 7 (upper)
    const int L = (warp & 3) * 32 + lane, hf = warp >> 2;
    const bool lower = L < 64;
    const int t = L & 63;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        sBad = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tslot;
    const uint32_t aKQ = smem_u32(sm + O_KQ), aRO = smem_u32(sm + O_RO), aS = smem_u32(sm + O_S),
                   aDS = smem_u32(sm + O_DS), aT = smem_u32(sm + O_T), aA = smem_u32(sm + O_A),
                   aR = smem_u32(sm + O_R), aU = smem_u32(sm + O_U), aDU = smem_u32(sm + O_DU);
    int mph = 0;   // phase of bar_mma
    auto mma_wait = [&]() {
        if (!mbar_wait(&bar_mma, (uint32_t)(mph & 1))) sBad = 1;
        ++mph;
        tc_fence_after();
    };

    // ---- loads: K, Q, dO, V (token rows), T, A^T (chunk slot), g, and the
    //      recorded bf16 tiles of S (rows i) and dS'^T (rows j), 32 KB each
    if (tid == 0) {
        mbar_expect_tx(&bar_ld, 10u * SL + 256u + 65536u);
        bulk_load(sm + O_S, S_img + slot * 32768, 32768u, &bar_ld);
        bulk_load(sm + O_DS, dS_img + slot * 32768, 32768u, &bar_ld);
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
            tma_load_3d(sm + O_KQ + s2 * 2 * SL, &mk, &bar_ld, 64 * s2, h, (int)row0);
            tma_load_3d(sm + O_KQ + s2 * 2 * SL + SL, &mq, &bar_ld, 64 * s2, h, (int)row0);
            tma_load_3d(sm + O_RO + s2 * 2 * SL + SL, &mo, &bar_ld, 64 * s2, h, (int)row0);
            tma_load_3d(sm + O_V + s2 * SL, &mv, &bar_ld, 64 * s2, h, (int)row0);
        }
        tma_load_2d(sm + O_T, &mt, &bar_ld, 0, (int)(slot * C));
        tma_load_2d(sm + O_A, &ma, &bar_ld, 0, (int)(slot * C));
        bulk_load(vg, g_ws + slot * C, 256u, &bar_ld);
    }
    if (tid < C) {
        const bool ok = tid < nc;
        const size_t r = (size_t)(row0 + tid) * p.H + h;
        valpha[tid] = (ok && p.alpha) ? p.alpha[r] : 1.f;
        veta[tid] = ok ? p.eta[r] : 0.f;
    }
    if (!mbar_wait(&bar_ld, 0u)) sBad = 1;
    // ---- sum of S o dS' (the dg_C term): row i of S, column i of dS'^T,
    //      the half jq of the columns j
    float sds = 0.f;
    {
        const int i = tid >> 1, jq = tid & 1;
        const unsigned char *srow = sm + O_S + jq * 16 * KB;
        const unsigned char *dcol = sm + O_DS + (i >> 6) * 16 * KB;
#pragma unroll 2
        for (int c8 = 0; c8 < 8; ++c8) {
            const uint4 w = *reinterpret_cast<const uint4 *>(srow + sw128_offset(i, 8 * c8));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 64 * jq + 8 * c8 + 2 * e;
                sds = fmaf(g_lo(ww[e]), g_at(dcol, j, i & 63), sds);
                sds = fmaf(g_hi(ww[e]), g_at(dcol, j + 1, i & 63), sds);
            }
        }
    }
    // ---- rows past the sequence's end: K, Q, dO, V cleared; chunk vectors
    if (nc < C) {
        for (int e = tid; e < (C - nc) * 16; e += NTH) {
            const int tt = nc + (e >> 4), pc = e & 15, s2 = pc >> 3;
            const uint32_t off = sw128_offset(tt, 8 * (pc & 7));
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(sm + O_KQ + s2 * 2 * SL + off) = z;
            *reinterpret_cast<uint4 *>(sm + O_KQ + s2 * 2 * SL + SL + off) = z;
            *reinterpret_cast<uint4 *>(sm + O_RO + s2 * 2 * SL + SL + off) = z;
            *reinterpret_cast<uint4 *>(sm + O_V + s2 * SL + off) = z;
        }
    }
    __syncthreads();
    {   // ||k_t||^2: four threads per row t = tid / 4, 32 features each
        const int tr = tid >> 2, part = tid & 3;
        const unsigned char *krow = sm + O_KQ + (part >> 1) * 2 * SL;
        float n2 = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
            const uint4 w = *reinterpret_cast<const uint4 *>(krow + sw128_offset(tr, 32 * (part & 1) + 8 * c8));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                n2 = fmaf(g_lo(ww[e]), g_lo(ww[e]), n2);
                n2 = fmaf(g_hi(ww[e]), g_hi(ww[e]), n2);
            }
        }
        n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
        n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
        if (part == 0) {
            const float den = n2 + p.eps;
            vden[tr] = den;
            const float b = p.beta_mode ? veta[tr] : (den != 0.f ? veta[tr] / den : 0.f);
            vbeta[tr] = tr < nc ? b : 0.f;
            veg[tr] = __expf(vg[tr]);
            vegc[tr] = __expf(vg[C - 1] - vg[tr]);
            vdg[tr] = 0.f;
        }
    }
    fence_async_smem();
    __syncthreads();

    // ================= phase 1
    if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_mn = idesc_bf16_f32(128, 128, false, true);
        constexpr uint32_t id_k128 = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t id_kk = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)   // K S: B = S read MN-major (n = j, k = i)
            mma_bf16(tb + C_A, gk_desc(aKQ, ks, 2 * SL), gm_desc(aS, ks, 16 * KB), id_mn, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)   // A_qk^T dO: A = A^T rows t, B = dO (n = j, k = s)
            mma_bf16(tb + C_B, gk_desc(aA, ks, 0), gm_desc(aRO + SL, ks, 2 * SL), id_mn, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)   // K dS': B = dS'^T rows j (K-major)
            mma_bf16(tb + C_C, gk_desc(aKQ, ks, 2 * SL), gk_desc(aDS, ks, 16 * KB), id_k128, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)   // [K ; Q] K^T
            mma_bf16(tb + C_G, gk_desc(aKQ, ks, 2 * SL), gk_desc(aKQ, ks, 2 * SL), id_kk, ks > 0);
        mma_commit(&bar_mma);
    }
    __syncwarp();
    mma_wait();
    // ---- epilogue 1 (rows t of the lower lanes): R and dU to bf16 tiles
    if (lower) {
        const float et = veg[t], ec = vegc[t], bt = vbeta[t];
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            const int j0 = 64 * hf + 32 * c2;
            uint32_t ks_[32], da[32], db[32];
            tmem_ld32(tb + lane_base + C_A + j0, ks_);
            tmem_ld32(tb + lane_base + C_B + j0, da);
            tmem_ld32(tb + lane_base + C_C + j0, db);
            tmem_ld_wait();
            float rr[32], uu[32];
            const unsigned char *vs = sm + O_V + hf * SL;
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const float v = g_at(vs, t, 32 * c2 + x);
                rr[x] = bt * (v - et * __uint_as_float(ks_[x]));
                uu[x] = fmaf(ec, __uint_as_float(db[x]), __uint_as_float(da[x]));
            }
            g_st16(sm + O_R + hf * SL, t, 32 * c2, rr);
            g_st16(sm + O_R + hf * SL, t, 32 * c2 + 16, rr + 16);
            g_st16(sm + O_DU + hf * SL, t, 32 * c2, uu);
            g_st16(sm + O_DU + hf * SL, t, 32 * c2 + 16, uu + 16);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ================= phase 2
    if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_u = idesc_bf16_f32(128, 128, false, true);
        constexpr uint32_t id_r = idesc_bf16_f32(128, 128, true, true);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)   // U = T R: A = T rows t, B = R (n = j, k = s)
            mma_bf16(tb + C_B, gk_desc(aT, ks, 0), gm_desc(aR, ks, SL), id_u, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)   // dR = T^T dU: A = T read MN-major (m = t, k = s)
            mma_bf16(tb + C_C, gm_desc(aT, ks, SL), gm_desc(aDU, ks, SL), id_r, ks > 0);
        mma_commit(&bar_mma);
    }
    __syncwarp();
    mma_wait();
    // ---- epilogue 2 (lower lanes): U, dR to bf16 tiles; dV; dbeta and dg from R
    if (lower) {
        const float et = veg[t], bt = vbeta[t];
        float p1 = 0.f, p2 = 0.f;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            const int j0 = 64 * hf + 32 * c2;
            uint32_t ur[32], rr[32], kr[32];
            tmem_ld32(tb + lane_base + C_B + j0, ur);
            tmem_ld32(tb + lane_base + C_C + j0, rr);
            tmem_ld32(tb + lane_base + C_A + j0, kr);
            tmem_ld_wait();
            float uf[32], df[32], dv[32];
            const unsigned char *vs = sm + O_V + hf * SL;
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                uf[x] = __uint_as_float(ur[x]);
                df[x] = __uint_as_float(rr[x]);
                dv[x] = bt * df[x];
                const float v = g_at(vs, t, 32 * c2 + x);
                p1 = fmaf(v - et * __uint_as_float(kr[x]), df[x], p1);   // (V - e^g K S) . dR
                p2 = fmaf(v, df[x], p2);
            }
            g_st16(sm + O_U + hf * SL, t, 32 * c2, uf);
            g_st16(sm + O_U + hf * SL, t, 32 * c2 + 16, uf + 16);
            g_st16(sm + O_RO + hf * 2 * SL, t, 32 * c2, df);   // dR: first tile of the pair
            g_st16(sm + O_RO + hf * 2 * SL, t, 32 * c2 + 16, df + 16);
            g_st16(sm + O_R + hf * SL, t, 32 * c2, dv);        // dV staging (R is read)
            g_st16(sm + O_R + hf * SL, t, 32 * c2 + 16, dv + 16);
        }
        vp[hf * 64 + t] = p1;
        vp[128 + hf * 64 + t] = p2;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid < C) {
        const float p1 = vp[tid] + vp[64 + tid], p2 = vp[128 + tid] + vp[192 + tid];
        vdbeta[tid] = p1;
        vdg[tid] += vbeta[tid] * (p1 - p2);   // -beta e^g (K S)_t . dR_t
    }
    // dV: TMA store of a whole chunk; a partial chunk row by row
    {
        __nv_bfloat16 *dvo = static_cast<__nv_bfloat16 *>(p.dv);
        if (nc == C) {
            if (tid == 0) {
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2)
                    tma_store_3d(&mdv, sm + O_R + s2 * SL, 64 * s2, h, (int)row0);
                bulk_commit_group();
            }
        } else {
            for (int e = tid; e < nc * 128; e += NTH) {
                const int tt = e >> 7, j = e & 127;
                dvo[((size_t)(row0 + tt) * p.H + h) * 128 + j] =
                    *reinterpret_cast<const __nv_bfloat16 *>(sm + O_R + (j >> 6) * SL + sw128_offset(tt, j & 63));
            }
        }
    }

    // ================= phase 3
    if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_64 = idesc_bf16_f32(128, 64, false, false);
        constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t id_umn = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)   // [dR ; dO] U^T: B = U rows s (K-major)
            mma_bf16(tb + C_A, gk_desc(aRO, ks, 2 * SL), gk_desc(aU, ks, SL), id_64, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)   // U dS'^T: B = dS'^T read MN-major (n = i, k = j)
            mma_bf16(tb + C_B, gk_desc(aU, ks, SL), gm_desc(aDS, ks, 16 * KB), id_umn, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)   // [dR ; dO] S^T
            mma_bf16(tb + C_C, gk_desc(aRO, ks, 2 * SL), gk_desc(aS, ks, 16 * KB), id_kk, ks > 0);
        mma_commit(&bar_mma);
    }
    __syncwarp();
    mma_wait();
    // the dV store has read the staging tile before [X + X^T | M1] overwrites
    // it; dbeta and dg of epilogue 2 are in place before the adds below
    if (tid == 0) bulk_wait_group_read0();
    __syncthreads();
    // ---- epilogue 3: lower lanes row t of dR U^T -> X and the dA_kk terms;
    //      upper lanes row t of dO U^T -> M1 = dA_qk o Gamma and its terms.
    //      fp32 64 x 64 scratch with rows EL floats apart (a thread writes its
    //      row in 16-byte pieces; the 8 rows of a quarter warp fall in 8
    //      different bank groups): E_qk and E_kk for the column sums in the
    //      dS'^T, T and A^T tiles, X in the S tile (all read by the products).
    constexpr int EL = 68;
    static_assert(2 * 64 * EL * 4 <= O_R - O_DS && 64 * EL * 4 <= O_DS - O_S, "scratch");
    float *Eqk = reinterpret_cast<float *>(sm + O_DS);
    float *Ekk = Eqk + 64 * EL;
    float *Xs = reinterpret_cast<float *>(sm + O_S);
    {
        const float gt = vg[t];
        const int s0 = 32 * hf;
        uint32_t dr[32], gr[32];
        tmem_ld32(tb + lane_base + C_A + s0, dr);   // dR U^T (lower) / dO U^T (upper)
        tmem_ld32(tb + lane_base + C_G + s0, gr);   // K K^T (lower) / Q K^T (upper)
        tmem_ld_wait();
        float rsum = 0.f, bsum = 0.f;
        if (lower) {
            const float bt = vbeta[t];
            float xrow[32], erow[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const int s2 = s0 + x;
                const float xg = s2 < t ? -__uint_as_float(dr[x]) * __expf(gt - vg[s2]) : 0.f;
                const float e = xg * __uint_as_float(gr[x]);   // . k_t k_s
                bsum += e;
                erow[x] = bt * e;                              // dA_kk o A_kk
                xrow[x] = bt * xg;                             // X
            }
            rsum = bt * bsum;
#pragma unroll
            for (int x = 0; x < 32; x += 4) {
                *reinterpret_cast<float4 *>(Ekk + t * EL + s0 + x) =
                    make_float4(erow[x], erow[x + 1], erow[x + 2], erow[x + 3]);
                *reinterpret_cast<float4 *>(Xs + t * EL + s0 + x) =
                    make_float4(xrow[x], xrow[x + 1], xrow[x + 2], xrow[x + 3]);
            }
        } else {
            float m1[32], erow[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const int s2 = s0 + x;
                const float da = s2 <= t ? __uint_as_float(dr[x]) * __expf(gt - vg[s2]) : 0.f;
                m1[x] = da;                                    // dA_qk o Gamma
                erow[x] = da * __uint_as_float(gr[x]);         // dA_qk o A_qk
                rsum += erow[x];
            }
#pragma unroll
            for (int x = 0; x < 32; x += 4)
                *reinterpret_cast<float4 *>(Eqk + t * EL + s0 + x) =
                    make_float4(erow[x], erow[x + 1], erow[x + 2], erow[x + 3]);
            g_st16(sm + O_R + SL, t, s0, m1);                  // M1 tile [t][s]
            g_st16(sm + O_R + SL, t, s0 + 16, m1 + 16);
        }
        // row sums of the two halves (both threads of a row add into vdg / vdbeta)
        atomicAdd(&vdg[t], rsum);
        if (lower) atomicAdd(&vdbeta[t], bsum);
    }
    __syncthreads();
    {   // column sums: dg_s -= sum_r E_qk[r][s] + E_kk[r][s]; four threads per
        // column s = tid % 64, 16 rows each
        const int sc = tid & 63, q = tid >> 6;
        float c0 = 0.f, c1 = 0.f;
#pragma unroll
        for (int r = 16 * q; r < 16 * q + 16; r += 2) {
            c0 += Eqk[r * EL + sc] + Ekk[r * EL + sc];
            c1 += Eqk[(r + 1) * EL + sc] + Ekk[(r + 1) * EL + sc];
        }
        vp[q * 64 + sc] = c0 + c1;   // (the half partials of epilogue 2 are consumed)
    }
    __syncthreads();
    if (tid < C) vdg[tid] -= (vp[tid] + vp[64 + tid]) + (vp[128 + tid] + vp[192 + tid]);
    {   // X + X^T (symmetric) to the first tile of the pair; zeros (8 KB) in U.
        // Row r = tid % 64 (consecutive lanes: the column reads are contiguous,
        // the row reads 16-byte pieces in 8 bank groups), columns 16 q .. + 15
        const int r = tid & 63, q = tid >> 6;
        float xx[16];
#pragma unroll
        for (int x = 0; x < 16; x += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(Xs + r * EL + 16 * q + x);
            xx[x] = a4.x + Xs[(16 * q + x) * EL + r];
            xx[x + 1] = a4.y + Xs[(16 * q + x + 1) * EL + r];
            xx[x + 2] = a4.z + Xs[(16 * q + x + 2) * EL + r];
            xx[x + 3] = a4.w + Xs[(16 * q + x + 3) * EL + r];
        }
        g_st16(sm + O_R, r, 16 * q, xx);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(sm + O_U + r * 128 + 32 * q) = z;
        *reinterpret_cast<uint4 *>(sm + O_U + r * 128 + 32 * q + 16) = z;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ================= phase 4
    if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_k = idesc_bf16_f32(128, 128, false, true);
        constexpr uint32_t id_q = idesc_bf16_f32(128, 128, true, true);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)   // [X + X^T ; M1] K: B = K read MN-major (n = i, k = s)
            mma_bf16(tb + C_A, gk_desc(aR, ks, 0), gm_desc(aKQ, ks, 2 * SL), id_k, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)   // + [M1^T ; 0] Q: A = M1 read MN-major, zeros beyond
            mma_bf16(tb + C_A, gm_desc(aR + SL, ks, aU - (aR + SL)), gm_desc(aKQ + SL, ks, 2 * SL),
                     id_q, 1);
        mma_commit(&bar_mma);
    }
    __syncwarp();
    mma_wait();
    // ---- final epilogue: dK (lower lanes), dQ (upper lanes), their dg terms
    __nv_bfloat16 *dqo = static_cast<__nv_bfloat16 *>(p.dq), *dko = static_cast<__nv_bfloat16 *>(p.dk);
    float red = 0.f;
    {
        const float et = veg[t], ec = vegc[t], bt = vbeta[t];
        float cn = 0.f;   // the gradient through beta's key norm
        if (lower && p.beta_mode == 0 && vden[t] != 0.f)
            cn = -2.f * veta[t] * vdbeta[t] / (vden[t] * vden[t]);
        float acc = 0.f;   // k . (U dS'^T)_t (lower) or q . pq_t (upper)
        unsigned char *stg = lower ? sm + O_S : sm + O_DU;   // staging: dK in S, dQ in dU
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            const int i0 = 64 * hf + 32 * c2;
            uint32_t ar[32], br[32], cr[32];
            tmem_ld32(tb + lane_base + C_C + i0, ar);   // dR S^T (lower) / pq (upper)
            tmem_ld32(tb + lane_base + C_A + i0, cr);   // (X + X^T) K + M1^T Q / M1 K
            if (lower) tmem_ld32(tb + lane_base + C_B + i0, br);   // U dS'^T
            tmem_ld_wait();
            float out[32];
            const unsigned char *ks_ = sm + O_KQ + hf * 2 * SL + (lower ? 0 : SL);   // k_t or q_t
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const float kv = g_at(ks_, t, 32 * c2 + x);
                if (lower) {
                    const float uds = __uint_as_float(br[x]);
                    out[x] = -bt * et * __uint_as_float(ar[x]) + ec * uds + __uint_as_float(cr[x]) + cn * kv;
                    acc = fmaf(kv, uds, acc);
                } else {
                    const float pq = __uint_as_float(ar[x]);
                    out[x] = et * pq + __uint_as_float(cr[x]);
                    acc = fmaf(kv, pq, acc);
                }
            }
            g_st16(stg + hf * SL, t, 32 * c2, out);
            g_st16(stg + hf * SL, t, 32 * c2 + 16, out + 16);
        }
        if (lower) {
            const float wk = ec * acc;
            atomicAdd(&vdg[t], -wk);
            red = wk;
        } else {
            atomicAdd(&vdg[t], et * acc);
        }
    }
    fence_async_smem();
    red += __shfl_xor_sync(0xffffffffu, red, 16);
    red += __shfl_xor_sync(0xffffffffu, red, 8);
    red += __shfl_xor_sync(0xffffffffu, red, 4);
    red += __shfl_xor_sync(0xffffffffu, red, 2);
    red += __shfl_xor_sync(0xffffffffu, red, 1);
    // S o dS' partial sums of the conversion, reduced per warp
    float sw = sds;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, off);
    if (lane == 0) vred[warp] = red + sw * veg[C - 1];
    tc_fence_before();
    __syncthreads();
    if (nc == C) {
        if (tid == 0) {
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                tma_store_3d(&mdk, sm + O_S + s2 * SL, 64 * s2, h, (int)row0);
                tma_store_3d(&mdq, sm + O_DU + s2 * SL, 64 * s2, h, (int)row0);
            }
            bulk_commit_group();
        }
    } else {
        for (int e = tid; e < nc * 128; e += NTH) {
            const int tt = e >> 7, i = e & 127;
            const uint32_t off = (i >> 6) * SL + sw128_offset(tt, i & 63);
            const size_t o = ((size_t)(row0 + tt) * p.H + h) * 128 + i;
            dko[o] = *reinterpret_cast<const __nv_bfloat16 *>(sm + O_S + off);
            dqo[o] = *reinterpret_cast<const __nv_bfloat16 *>(sm + O_DU + off);
        }
    }
    if (warp == 0) {   // dg_C onto g_{C-1}; reverse cumulative sum -> dlog(alpha)
        float gc = 0.f;
#pragma unroll
        for (int w = 0; w < NTH / 32; ++w) gc += vred[w];
        float d0 = vdg[lane], d1 = vdg[lane + 32];
        if (lane == 31) d1 += gc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {   // suffix sums
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
                if (p.dalpha && p.alpha) p.dalpha[r] = dl[q2] / valpha[tt];
                if (p.deta) {
                    const float dbt = vdbeta[tt], den = vden[tt];
                    p.deta[r] = p.beta_mode ? dbt : (den != 0.f ? dbt / den : 0.f);
                }
            }
        }
    }
    if (tid == 0) {
        bulk_wait_group0();
        if (sBad && p.status) atomicCAS(p.status, 0u, kDevTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// Varlen: validates cu_seqlens (cu[0] == 0, non-decreasing, cu[N] ==
// total_T; a bad table sets the status word and every later kernel of the
// call skips its work) and builds the chunk tables: the first chunk of each
// sequence (chunk_prefix[N + 1]) and the sequence of each chunk (chunk_seq).
constexpr int BP_THREADS = 1024;

__global__ void __launch_bounds__(BP_THREADS)
bwd_prep_kernel(const int *cu, int N, int total_T, int *chunk_prefix, int *chunk_seq,
                unsigned *status) {
    __shared__ int bad, carry;
    __shared__ int warp_sums[BP_THREADS / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        bad = (cu[0] != 0 || cu[N] != total_T) ? 1 : 0;
        carry = 0;
    }
    __syncthreads();
    for (int i = tid; i < N; i += BP_THREADS)
        if (cu[i + 1] < cu[i]) atomicOr(&bad, 1);
    __syncthreads();
    if (bad) {
        if (tid == 0) *status = kDevBadSeqlens;
        return;
    }
    // exclusive prefix sum of the chunk counts, BP_THREADS sequences at a time
    for (int base = 0; base < N; base += BP_THREADS) {
        const int n = base + tid;
        const int cnt = n < N ? (cu[n + 1] - cu[n] + C - 1) / C : 0;
        int x = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp ? warp_sums[warp - 1] : 0) + carry;
        if (n < N) chunk_prefix[n] = incl - cnt;
        __syncthreads();
        if (tid == BP_THREADS - 1) carry = incl;
        __syncthreads();
    }
    if (tid == 0) chunk_prefix[N] = carry;
    __syncthreads();
    for (int n = 0; n < N; ++n) {   // sequences in order; their chunks in parallel
        const int c0 = chunk_prefix[n], c1 = chunk_prefix[n + 1];
        for (int g = c0 + tid; g < c1; g += BP_THREADS) chunk_seq[g] = n;
    }
}

long bwd_chunks(bool varlen, int n_seq, int T, int total_T) {
    // every varlen sequence adds at most one partial chunk
    return varlen ? ((long)total_T + C - 1) / C + n_seq : (long)n_seq * ((T + C - 1) / C);
}

// bf16 with d = 128 and at least one 64-row TMA box: the tensor-core forward
// records the chunk-start states, and the dS chain reads its chunk workspace.
bool bwd_uses_tc(long total_T, int d, int dtype) {
    return chunk_tc_supported(d, dtype) && total_T >= C;
}

struct BwdLayout {
    size_t tables, S, dS, Tm, tc, total;
};
BwdLayout bwd_layout(bool varlen, int n_seq, int T, int total_T, int H, int d, int dtype) {
    const long nchunks = bwd_chunks(varlen, n_seq, T, total_T);
    BwdLayout L;
    L.tables = 0;
    const size_t tab = varlen ? ((size_t)n_seq + 1 + (size_t)nchunks) * sizeof(int) : 0;
    L.S = (tab + 255) / 256 * 256;
    const bool tc = bwd_uses_tc(total_T, d, dtype);
    // S and dS' per chunk slot: fp32 [d][d], or on the tensor-core path the
    // two 32 KB bf16 tile images
    const size_t per = tc ? 32768 : (size_t)d * d * sizeof(float);
    L.dS = L.S + (size_t)nchunks * H * per;
    L.Tm = L.dS + (size_t)nchunks * H * per;
    // tensor-core path: T (bf16) of every chunk slot, then the forward's workspace
    L.tc = L.Tm + (tc ? ((size_t)nchunks * H * C * C * 2 + 1023) / 1024 * 1024 : 0);
    L.total = L.tc + (tc ? chunk_tc_workspace_bytes(nchunks, H, n_seq) : 0);
    return L;
}

template <typename Tin, int D>
cudaError_t launch_bwd_t(const BwdProblem &p0, cudaStream_t s) {
    const bool varlen = p0.cu_seqlens != nullptr;
    const long nchunks = bwd_chunks(varlen, p0.n_seq, p0.T, p0.total_T);
    const int nch_fixed = varlen ? 0 : (p0.T + C - 1) / C;
    const int units = p0.n_seq * p0.H;
    const BwdLayout L = bwd_layout(varlen, p0.n_seq, p0.T, p0.total_T, p0.H, D, p0.dtype);
    unsigned char *ws = static_cast<unsigned char *>(p0.ws);
    BwdProblem p = p0;
    cudaError_t e;
    if (varlen) {
        int *prefix = reinterpret_cast<int *>(ws + L.tables);
        p.chunk_prefix = prefix;
        p.chunk_seq = prefix + p0.n_seq + 1;
        bwd_prep_kernel<<<1, BP_THREADS, 0, s>>>(p0.cu_seqlens, p0.n_seq, p0.total_T, prefix,
                                                  prefix + p0.n_seq + 1, p0.status);
        note_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    float *S_chk = reinterpret_cast<float *>(ws + L.S);
    float *dS_chk = reinterpret_cast<float *>(ws + L.dS);
    const bool tc = bwd_uses_tc(p0.total_T, D, p0.dtype);
    // 1. states at the chunk starts (the forward, no outputs)
    Problem f{};
    f.q = p.q; f.k = p.k; f.v = p.v; f.alpha = p.alpha; f.eta = p.eta; f.eps = p.eps;
    f.S0 = p.S0; f.o = nullptr; f.S_T = nullptr; f.cu_seqlens = p.cu_seqlens;
    f.n_seq = p.n_seq; f.T = varlen ? 0 : p.T; f.total_T = p.total_T; f.H = p.H; f.d = D;
    f.dtype = p.dtype; f.beta_mode = p.beta_mode; f.S_chk = S_chk; f.status = p.status;
    f.chunk_prefix = p.chunk_prefix;
    float *g_ws = nullptr;
    void *W_ws = nullptr, *A_ws = nullptr;
    if (tc) {
        f.T_chk = ws + L.Tm;
        f.ws = ws + L.tc;
        f.ws_bytes = L.total - L.tc;
        chunk_tc_ws_views(f.ws, nchunks, p.H, p.n_seq, &g_ws, &W_ws, &A_ws);
        // the single-launch form's ready flags start at zero
        const size_t reset = chunk_tc_reset_bytes(f, nchunks);
        if (reset > 0 && (e = cudaMemsetAsync(f.ws, 0, reset, s)) != cudaSuccess) return e;
        e = launch_chunk_tc(f, nchunks, s);
    } else {
        e = launch_chunk_simt(f, s);
    }
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
        if ((e = cudaFuncSetAttribute(bwd_dstate_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)dtc::SMEM)) != cudaSuccess)
            return e;
        attr = true;
    }
    if (tc) {
        CUtensorMap mq, mk, mo, mw, ma;
        const long slots = nchunks * p.H;
        if (!tmap::rows_3d(&mq, p.q, p.H, p.total_T, C) || !tmap::rows_3d(&mk, p.k, p.H, p.total_T, C) ||
            !tmap::rows_3d(&mo, p.dout, p.H, p.total_T, C) ||
            !tmap::plain_2d(&mw, W_ws, D, slots * C, C) || !tmap::plain_2d(&ma, A_ws, C, slots * C, C))
            return cudaErrorInvalidValue;
        bwd_dstate_tc_kernel<<<units, dtc::THREADS, dtc::SMEM, s>>>(
            mq, mk, mo, mw, ma, p, reinterpret_cast<unsigned char *>(dS_chk), g_ws);
    } else {
        bwd_dstate_kernel<Tin, D><<<dim3(units, D / DVB), NT, sizeof(DsSmem<D>), s>>>(p, dS_chk);
    }
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3. token gradients, one CTA per chunk slot
    if (tc) {
        static bool gattr = false;
        if (!gattr) {
            if ((e = cudaFuncSetAttribute(bwd_grads_tc_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)gtc::SMEM)) != cudaSuccess)
                return e;
            gattr = true;
        }
        CUtensorMap mq, mk, mv, mo, mt, ma, mdq, mdk, mdv;
        const long slots = nchunks * p.H;
        if (!tmap::rows_3d(&mq, p.q, p.H, p.total_T, C) || !tmap::rows_3d(&mk, p.k, p.H, p.total_T, C) ||
            !tmap::rows_3d(&mv, p.v, p.H, p.total_T, C) ||
            !tmap::rows_3d(&mo, p.dout, p.H, p.total_T, C) ||
            !tmap::plain_2d(&mt, f.T_chk, C, slots * C, C) ||
            !tmap::plain_2d(&ma, A_ws, C, slots * C, C) ||
            !tmap::rows_3d(&mdq, p.dq, p.H, p.total_T, C) ||
            !tmap::rows_3d(&mdk, p.dk, p.H, p.total_T, C) ||
            !tmap::rows_3d(&mdv, p.dv, p.H, p.total_T, C))
            return cudaErrorInvalidValue;
        bwd_grads_tc_kernel<<<dim3((unsigned)nchunks, p.H), gtc::NTH, gtc::SMEM, s>>>(
            mq, mk, mv, mo, mt, ma, mdq, mdk, mdv, p, nch_fixed,
            reinterpret_cast<const unsigned char *>(S_chk), reinterpret_cast<const unsigned char *>(dS_chk),
            g_ws);
    } else {
        bwd_grads_kernel<Tin, D><<<dim3((unsigned)nchunks, p.H), NT, sizeof(GrSmem<D>), s>>>(
            p, nch_fixed, S_chk, dS_chk);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace

size_t chunk_bwd_workspace_bytes(bool varlen, int n_seq, int T, int total_T, int H, int d,
                                 int dtype) {
    return bwd_layout(varlen, n_seq, T, total_T, H, d, dtype).total;
}

cudaError_t launch_chunk_bwd(const BwdProblem &p, cudaStream_t s) {
    if (p.n_seq == 0 || p.total_T == 0) return cudaSuccess;
    if (p.dtype == 1)
        return p.d == 128 ? launch_bwd_t<__nv_bfloat16, 128>(p, s)
                          : launch_bwd_t<__nv_bfloat16, 64>(p, s);
    return p.d == 128 ? launch_bwd_t<float, 128>(p, s) : launch_bwd_t<float, 64>(p, s);
}

}  // namespace kla
