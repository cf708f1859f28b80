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
// bf16 inputs with d = 128 take the tensor cores (section below): the query
// streams blocks of 128 tokens through tcgen05 products (Q K^T, K^T K and
// Q M + A' K) with the finish in the products' epilogue; M is carried in fp32
// and enters its product with Q rounded to bf16.
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

#include <algorithm>
#include <cstdint>

#include "kla_internal.h"
#include "kla_tc.cuh"
#include "kla_tmap.h"

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
//
// Per (sequence, head) the tokens go in blocks of NB = 128.  With M_b, m_b
// the statistics before block b and, for token t of the block,
//   s_t = (m_t . q_t) / n_t = (m_b . q_t + sum_{s<=t} q_t . k_s) / n_t,
//   M_t q_t - s_t m_t = (Q M_b)_t - s_t m_b + sum_{s<=t} (q_t . k_s - s_t) k_s,
// so with G = Q K^T and A'_ts = G_ts - s_t for s <= t (0 above the diagonal)
//   O = Q M_b + A' K,   q_clean_t = q_t - lambda_t / n_t (O_t - s_t m_b),
// and M_{b+1} = M_b + K^T K, m_{b+1} = m_b + the block's key sums.  No product
// waits for another block's output: the only carried quantities are M and m,
// so the blocks stream through the tensor cores and the finish is the
// products' epilogue.
//
// ccq_query_tc_kernel: one CTA per (sequence, head, segment); a loader warp
// (TMA, two stages of Q and K), an MMA warp and sixteen main warps.  M lives
// in TMEM (fp32): it starts as the initial statistics, and the K^T K of every
// block before the segment is added first (the prefix: keys only, two blocks
// per stage), then the segment's blocks in order.  Per block of the segment the MMA warp issues
// G = Q K^T, then M += K^T K once the main warps have copied M_b to shared
// memory (bf16), then O = Q M_b + A' K once they have written A' (bf16 pairs
// in TMEM).  Main thread (row L, 32-column group cg) forms the row's part of
// s_t and of A', finishes its part of row L of the previous block from O
// (staged in shared memory, stored by TMA) and copies its part of row L of M
// for the next block.  Segments are cut so that prefix and own blocks cost about the
// same in every CTA (a prefix block, keys only, costs about a quarter of a
// segment block).
namespace ctc {
constexpr int D = 128;
constexpr int NB = 128;                        // tokens per block
constexpr uint32_t SLAB = 128u * 128u;         // 128 rows x 64 bf16, 128-byte swizzle
constexpr uint32_t TILE = 2u * SLAB;           // 128 x 128 bf16: two 64-column slabs
constexpr int NST = 2;                         // stages: Q and K of one block each
constexpr uint32_t ST_Q = 0, ST_K = TILE, ST_BYTES = 2u * TILE;
constexpr uint32_t SM_M = NST * ST_BYTES;      // M_b (bf16; B operand of Q M_b)
constexpr uint32_t SM_OUT = SM_M + TILE;       // q_clean of a block (bf16), stored by TMA
constexpr uint32_t SM_F = SM_OUT + TILE;       // fp32 scratch:
constexpr uint32_t F_M = 0;                    //   m of three blocks [3][D]
constexpr int NMAIN = 16, THREADS = (NMAIN + 2) * 32;  // main warps: 4 lane quadrants x NCG
constexpr int NCG = NMAIN / 4, CW = D / NCG;   // column groups, columns per main thread
constexpr int RG = NMAIN * 32 / 16;            // token-row groups of the key sums
constexpr int FC_LD = D + 8;                   // row stride of the key-sum partials (the
                                               // four lanes of a feature hit four bank groups)
constexpr uint32_t F_X = F_M + 3 * D;          //   row partials of s_t [NCG][NB]
constexpr uint32_t F_C = F_X + NCG * NB;       //   key-sum partials, row groups paired [RG / 2][FC_LD]
constexpr uint32_t F_END = F_C + RG / 2 * FC_LD;
constexpr uint32_t SMEM = SM_F + F_END * 4 + 1024;   // + alignment slack
// TMEM columns: G = Q K^T, the fp32 statistics M (K^T K adds into it), the
// output product O, and A' (bf16 pairs) in two buffers of 64 columns
constexpr uint32_t TM_G = 0, TM_M = 128, TM_O = 256, TM_A = 384;
constexpr int P_MAX = 8;
constexpr float PREFIX_COST = 0.25f;           // a prefix block against a segment block
static_assert(SMEM <= 232448 - 1024, "shared memory of the CCQ kernel");
}  // namespace ctc

struct CcqTcParams {
    const float *lambda, *Ms0, *ms0, *ns0;
    float *Ms_T, *ms_T, *ns_T;
    unsigned *status;
    int T, H, P;
    int seg_start[ctc::P_MAX + 1];   // first block of each segment; seg_start[P] = blocks
};

__device__ __forceinline__ unsigned char *ccq_align1024(unsigned char *p) {
    const uint32_t a = tc::smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}
__device__ __forceinline__ void ccq_set_status(unsigned *status, unsigned code) {
    if (status) atomicCAS(status, 0u, code);
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);   // a -> low half
    return *reinterpret_cast<const uint32_t *>(&v);
}
// 16 fp32 values -> bf16 columns [c0, c0 + 16) of row `row` of a 64-column
// slab stored with the 128-byte swizzle.
__device__ __forceinline__ void st_row16(unsigned char *slab, int row, int c0, const uint32_t *r) {
#pragma unroll
    for (int k = 0; k < 2; ++k)
        *reinterpret_cast<uint4 *>(slab + tc::sw128_offset(row, c0 + 8 * k)) =
            make_uint4(pack_bf2(__uint_as_float(r[8 * k + 0]), __uint_as_float(r[8 * k + 1])),
                       pack_bf2(__uint_as_float(r[8 * k + 2]), __uint_as_float(r[8 * k + 3])),
                       pack_bf2(__uint_as_float(r[8 * k + 4]), __uint_as_float(r[8 * k + 5])),
                       pack_bf2(__uint_as_float(r[8 * k + 6]), __uint_as_float(r[8 * k + 7])));
}
// Barrier over `count` threads that also returns the OR of `pred` over them
// (the same answer in every thread).
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1 : 0), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}
// Operand descriptors for the 128 x 128 tiles: K-major (rows of 64-element
// slabs, the K step of 16 elements is 32 bytes inside a slab) and MN-major
// (K step of 16 rows = 2048 bytes; the two 64-element MN halves one slab
// apart).
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int ks) {
    return tc::sdesc_sw128(base + (uint32_t)(ks >> 2) * ctc::SLAB + (uint32_t)(ks & 3) * 32u, 16,
                           1024);
}
__device__ __forceinline__ uint64_t mdesc(uint32_t base, int ks) {
    return tc::sdesc_sw128(base + (uint32_t)ks * 2048u, ctc::SLAB, 1024);
}

// The items a CTA loads, in order: the npre prefix blocks (keys only) two to
// an item (the second block's keys in the stage's query half), then the
// segment's nb blocks (queries and keys); item i uses stage i % NST.
//
// Block n of the segment, in order on the tensor pipe:
//   G_{n+1} = Q K^T of the next block (once A'_n is in TMEM: G is read),
//   M += K_n^T K_n (once the main warps have copied M_n to shared memory),
//   O_n = Q M_n + A'_n K (A' from TMEM).
// The main warps, for block n: s_t and A'_n from G_n, then (after O_{n-1})
// the finish of block n - 1 and the copy of M_n; so A'_n is formed while
// O_{n-1} runs and G_{n+1} runs while block n - 1 is finished.
__global__ void __launch_bounds__(ctc::THREADS, 1)
ccq_query_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mo, const CcqTcParams p) {
    using namespace ctc;
    using namespace tc;
    extern __shared__ unsigned char ccq_smem[];
    unsigned char *sm = ccq_align1024(ccq_smem);
    __shared__ uint64_t bar_ld[NST], bar_empty[NST];
    __shared__ uint64_t bar_init, bar_pre, bar_g, bar_o, bar_a, bar_m, bar_fin;
    __shared__ uint32_t tslot;
    __shared__ int sAbort;
    unsigned char *sM = sm + SM_M, *sOut = sm + SM_OUT;
    float *fm = reinterpret_cast<float *>(sm + SM_F) + F_M;
    float *fx = reinterpret_cast<float *>(sm + SM_F) + F_X;
    float *fc = reinterpret_cast<float *>(sm + SM_F) + F_C;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x / p.P, seg = blockIdx.x % p.P;
    const int bq = unit / p.H, h = unit % p.H;
    const int npre = p.seg_start[seg];                  // prefix blocks
    const int npi = (npre + 1) / 2;                     // prefix items
    const int nb = p.seg_start[seg + 1] - npre;         // the segment's blocks

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&bar_ld[i], 1);
            mbar_init(&bar_empty[i], NMAIN + 1);   // the main warps' reads and the products
        }
        mbar_init(&bar_init, NMAIN);   // initial M in TMEM
        mbar_init(&bar_pre, 1);        // prefix products done
        mbar_init(&bar_g, 1);
        mbar_init(&bar_o, 1);
        mbar_init(&bar_a, NMAIN);      // one arrival per main warp
        mbar_init(&bar_m, NMAIN);
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
    if (pre_abort || nb <= 0) {
        if (warp == 0) tmem_dealloc(tb, 512);
        return;
    }
    auto fail = [&]() {
        *(volatile int *)&sAbort = 1;   // read by the other warps' waits
        ccq_set_status(p.status, kDevTimeout);
    };

    if (warp == NMAIN + 1) {
        // ------------------------------------------------------------ loader
        const int nitems = npi + nb;
        int i = 0;
        for (; i < nitems; ++i) {
            const int s = i % NST, k = i / NST;
            if (k >= 1 &&
                !__all_sync(0xffffffffu,
                            mbar_wait_or_abort(&bar_empty[s], (uint32_t)((k - 1) & 1), &sAbort))) {
                fail();
                break;
            }
            if (lane == 0) {
                unsigned char *st = sm + s * ST_BYTES;
                if (i >= npi) {   // block npre + (i - npi): queries and keys
                    const int tok0 = (npre + i - npi) * NB;
                    mbar_expect_tx(&bar_ld[s], 4u * 16384u);
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        tma_load_4d(st + ST_Q + sl * SLAB, &mq, &bar_ld[s], 64 * sl, h, tok0, bq);
                        tma_load_4d(st + ST_K + sl * SLAB, &mk, &bar_ld[s], 64 * sl, h, tok0, bq);
                    }
                } else {          // prefix blocks 2i and 2i + 1: keys only
                    const bool two = 2 * i + 1 < npre;
                    mbar_expect_tx(&bar_ld[s], (two ? 4u : 2u) * 16384u);
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        tma_load_4d(st + ST_K + sl * SLAB, &mk, &bar_ld[s], 64 * sl, h, 2 * i * NB, bq);
                        if (two)
                            tma_load_4d(st + ST_Q + sl * SLAB, &mk, &bar_ld[s], 64 * sl, h,
                                        (2 * i + 1) * NB, bq);
                    }
                }
            }
            __syncwarp();
        }
        // on an early exit the loads still in flight (one per stage at most)
        // land before the CTA leaves
        if (sAbort)
            for (int k = i > NST ? i - NST : 0; k < i; ++k)
                (void)mbar_wait(&bar_ld[k % NST], (uint32_t)((k / NST) & 1));
    } else if (warp == NMAIN) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t id_g = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t id_z = idesc_bf16_f32(128, 128, true, true);
        constexpr uint32_t id_o = idesc_bf16_f32(128, 128, false, true);
        const uint32_t aM = smem_u32(sM);
        auto aQ = [&](int i) { return smem_u32(sm + (i % NST) * ST_BYTES + ST_Q); };
        auto aK = [&](int i) { return smem_u32(sm + (i % NST) * ST_BYTES + ST_K); };
        // M += K^T K for the keys at shared address a (read MN-major for both operands)
        auto issue_z = [&](uint32_t a) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tb + TM_M, mdesc(a, ks), mdesc(a, ks), id_z, 1);
        };
        // G = Q K^T (both K-major) of item i into TMEM
        auto issue_g = [&](int i) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tb + TM_G, kdesc(aQ(i), ks), kdesc(aK(i), ks), id_g, ks > 0);
            mma_commit(&bar_g);
        };
        bool ok = true;
        // ---- prefix: the initial M is in TMEM, then K^T K of every block before the segment
        if (npre > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bar_init, 0u, &sAbort));
            for (int i = 0; ok && i < npi; ++i) {
                ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bar_ld[i % NST],
                                                                (uint32_t)((i / NST) & 1), &sAbort));
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    issue_z(aK(i));
                    if (2 * i + 1 < npre) issue_z(aQ(i));
                    mma_commit(&bar_empty[i % NST]);
                }
                __syncwarp();
            }
            if (ok && lane == 0) mma_commit(&bar_pre);
            __syncwarp();
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&bar_ld[npi % NST],
                                                                (uint32_t)((npi / NST) & 1), &sAbort));
        if (!ok) fail();
        if (ok) {
            tc_fence_after();
            if (lane == 0) issue_g(npi);
            __syncwarp();
        }
        for (int n = 0; ok && n < nb; ++n) {
            const int i = npi + n;
            // A'_n in TMEM (G_n read), and the next block landed: G_{n+1}
            bool w = mbar_wait_or_abort(&bar_a, (uint32_t)(n & 1), &sAbort);
            if (w && n + 1 < nb)
                w = mbar_wait_or_abort(&bar_ld[(i + 1) % NST], (uint32_t)(((i + 1) / NST) & 1),
                                       &sAbort);
            if (!__all_sync(0xffffffffu, w)) { fail(); break; }
            tc_fence_after();
            if (lane == 0 && n + 1 < nb) issue_g(i + 1);
            __syncwarp();
            // M_n copied out of TMEM: M += K_n^T K_n; then O_n = Q M_n + A'_n K
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_m, (uint32_t)(n & 1), &sAbort))) {
                fail();
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                issue_z(aK(i));
                const uint32_t tA = tb + TM_A + 64u * (uint32_t)(n & 1);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tb + TM_O, kdesc(aQ(i), ks), mdesc(aM, ks), id_o, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ts(tb + TM_O, tA + 8u * (uint32_t)ks, mdesc(aK(i), ks), id_o, 1);
                mma_commit(&bar_o);
                mma_commit(&bar_empty[i % NST]);   // the stage may be refilled
            }
            __syncwarp();
        }
        // every MMA issued has completed before the CTA releases its TMEM
        if (lane == 0) mma_commit(&bar_fin);
        __syncwarp();
        (void)mbar_wait(&bar_fin, 0u);
    } else {
        // ------------------------------------------------------------ main warps
        const int L = (warp & 3) * 32 + lane;   // TMEM lane: token row / row of M
        const int cg = warp >> 2, j0 = CW * cg; // column group: columns [j0, j0 + CW)
        const int cs = j0 & 63;                 // first column inside its 64-column slab
        unsigned char *const sMs = sM + (j0 >> 6) * SLAB;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tM = tb + lane_base + TM_M + (uint32_t)j0;
        const float n0 = p.ns0 ? p.ns0[unit] : 0.f;
        bool bad = false;            // a wait of this warp gave up
        // ---- the initial statistics: M in TMEM (and, without a prefix, as
        //      bf16 in shared memory for Q M_0)
        {
            const float *m0 = p.Ms0 ? p.Ms0 + ((size_t)unit * D + L) * D + j0 : nullptr;
            const bool v4 = m0 && (reinterpret_cast<uintptr_t>(m0) & 15u) == 0;
#pragma unroll 1
            for (int c4 = 0; c4 < CW / 16; ++c4) {
                uint32_t r[16];
                if (v4) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 v = reinterpret_cast<const float4 *>(m0 + 16 * c4)[i];
                        r[4 * i] = __float_as_uint(v.x); r[4 * i + 1] = __float_as_uint(v.y);
                        r[4 * i + 2] = __float_as_uint(v.z); r[4 * i + 3] = __float_as_uint(v.w);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(m0 ? m0[16 * c4 + i] : 0.f);
                }
                tmem_st16(tM + 16 * c4, r);
                if (npre == 0) st_row16(sMs, L, cs + 16 * c4, r);
            }
            tmem_st_wait();
            if (npre == 0) fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(npre > 0 ? &bar_init : &bar_m);
        }
        // ---- the prefix: key sums of the blocks before the segment (the
        //      products add their K^T K to M meanwhile)
        const int kc = tid & 15, krg = tid >> 4;   // 16-byte piece (features 8kc..), row group
        float ka[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        // adds rows krg, krg + RG, ... of the key tile at `kt` (two slabs)
        auto key_sums = [&](const unsigned char *kt) __attribute__((always_inline)) {
            const unsigned char *kb = kt + (kc >> 3) * SLAB;
#pragma unroll
            for (int i = 0; i < NB / RG; ++i) {
                const uint4 w = *reinterpret_cast<const uint4 *>(kb + sw128_offset(krg + RG * i, 8 * (kc & 7)));
                ka[0] += bf_lo(w.x); ka[1] += bf_hi(w.x); ka[2] += bf_lo(w.y); ka[3] += bf_hi(w.y);
                ka[4] += bf_lo(w.z); ka[5] += bf_hi(w.z); ka[6] += bf_lo(w.w); ka[7] += bf_hi(w.w);
            }
        };
        // row groups krg and krg ^ 1 (lanes l and l ^ 16) combined by a shuffle,
        // then one partial row per pair
        auto put_key_sums = [&]() __attribute__((always_inline)) {
#pragma unroll
            for (int x = 0; x < 8; ++x) ka[x] += __shfl_xor_sync(0xffffffffu, ka[x], 16);
            if ((krg & 1) == 0) {
                float4 *dst = reinterpret_cast<float4 *>(fc + (krg >> 1) * FC_LD + 8 * kc);
                dst[0] = make_float4(ka[0], ka[1], ka[2], ka[3]);
                dst[1] = make_float4(ka[4], ka[5], ka[6], ka[7]);
            }
#pragma unroll
            for (int x = 0; x < 8; ++x) ka[x] = 0.f;
        };
        // the sum over the partial rows of feature tid >> 2, by the four lanes
        // tid & ~3 .. tid | 3 (lane part: rows part, part + 4, ...); every main
        // thread calls it
        auto sum_key_sums = [&]() __attribute__((always_inline)) -> float {
            const int f = tid >> 2, part = tid & 3;
            float c = 0.f;
#pragma unroll
            for (int g = 0; g < RG / 8; ++g) c += fc[(part + 4 * g) * FC_LD + f];
            c += __shfl_xor_sync(0xffffffffu, c, 1);
            c += __shfl_xor_sync(0xffffffffu, c, 2);
            return c;
        };
        for (int i = 0; i < npi; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_ld[i % NST],
                                                            (uint32_t)((i / NST) & 1), &sAbort))) {
                bad = true;
                fail();
                break;
            }
            key_sums(sm + (i % NST) * ST_BYTES + ST_K);
            if (2 * i + 1 < npre) key_sums(sm + (i % NST) * ST_BYTES + ST_Q);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_empty[i % NST]);
        }
        put_key_sums();
        named_sync(1, NMAIN * 32);
        {
            const float c = sum_key_sums();
            if (tid < 4 * D && (tid & 3) == 0)
                fm[tid >> 2] = (p.ms0 ? p.ms0[(size_t)unit * D + (tid >> 2)] : 0.f) + c;
        }
        if (npre > 0) {
            // M_0 = the initial M plus the prefix's K^T K, to shared memory (bf16)
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_pre, 0u, &sAbort))) {
                bad = true;
                fail();
            }
            tc_fence_after();
#pragma unroll
            for (int c4 = 0; c4 < CW / 16; ++c4) {
                uint32_t r[16];
                tmem_ld16(tM + 16 * c4, r);
                tmem_ld_wait();
                st_row16(sMs, L, cs + 16 * c4, r);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_m);
        }
        // m_0 visible, the partials' rows free again
        const bool stop0 = named_sync_or(1, NMAIN * 32, bad);

        // what the finish of a block needs, carried to the next iteration
        float sp = 0.f, scale = 0.f; // s_t, lambda_t / n_t
        // q_clean of block n from O (TMEM) and q_t (registers), staged in
        // shared memory and stored by TMA (rows past the sequence's end are
        // not written)
        auto finish = [&](int n, const uint4 (&qp)[CW / 8]) __attribute__((always_inline)) {
            const uint32_t tO = tb + lane_base + TM_O + (uint32_t)j0;
            const float4 *mb4 = reinterpret_cast<const float4 *>(fm + (n % 3) * D + j0);
            unsigned char *so = sOut + (j0 >> 6) * SLAB;
#pragma unroll
            for (int c2 = 0; c2 < CW / 32; ++c2) {
                uint32_t rr[2][16];
                tmem_ld16(tO + 32 * c2, rr[0]);
                tmem_ld16(tO + 32 * c2 + 16, rr[1]);
                tmem_ld_wait();
#pragma unroll
                for (int c1 = 0; c1 < 2; ++c1) {
                    const int c4 = 2 * c2 + c1;
                    const uint32_t (&r)[16] = rr[c1];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint4 qk = qp[2 * c4 + k];
                        const uint32_t qw[4] = {qk.x, qk.y, qk.z, qk.w};
                        const float4 ma = mb4[4 * c4 + 2 * k], mc = mb4[4 * c4 + 2 * k + 1];
                        const float mv[8] = {ma.x, ma.y, ma.z, ma.w, mc.x, mc.y, mc.z, mc.w};
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int x = 8 * k + 2 * e;
                            const float o0 = __uint_as_float(r[x]) - sp * mv[2 * e];
                            const float o1 = __uint_as_float(r[x + 1]) - sp * mv[2 * e + 1];
                            w[e] = pack_bf2(bf_lo(qw[e]) - scale * o0, bf_hi(qw[e]) - scale * o1);
                        }
                        *reinterpret_cast<uint4 *>(so + sw128_offset(L, cs + 16 * c4 + 8 * k)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_async_smem();
            named_sync(3, NMAIN * 32);
            if (tid == 0) {
#pragma unroll
                for (int sl = 0; sl < 2; ++sl)
                    tma_store_4d(&mo, sOut + sl * SLAB, 64 * sl, h, (npre + n) * NB, bq);
                bulk_commit_group();
            }
        };
        // block n; qc receives q_t of block n, qp holds that of block n - 1.
        // Returns true when the CTA gives up.
        auto step = [&](int n, uint4 (&qc)[CW / 8], const uint4 (&qp)[CW / 8]) __attribute__((always_inline)) -> bool {
            const int i = npi + n;
            const unsigned char *st = sm + (i % NST) * ST_BYTES;
            const int tok = (npre + n) * NB + L;
            const float lam_n = tok < p.T ? p.lambda[((size_t)bq * p.T + tok) * p.H + h] : 0.f;
            bool ok = mbar_wait_or_abort(&bar_ld[i % NST], (uint32_t)((i / NST) & 1), &sAbort) &&
                      mbar_wait_or_abort(&bar_g, (uint32_t)(n & 1), &sAbort);
            if (!__all_sync(0xffffffffu, ok)) {
                bad = true;
                fail();
            }
            tc_fence_after();
            // ---- row part of s_t: sum_{s <= t} G_ts and m_b . q_t over the half
            const float *mb = fm + (n % 3) * D;
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int c2 = 0; c2 < CW / 32; ++c2) {
                uint32_t r[2][16];
                tmem_ld16(tb + lane_base + TM_G + j0 + 32 * c2, r[0]);
                tmem_ld16(tb + lane_base + TM_G + j0 + 32 * c2 + 16, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    rs0 += (j0 + 32 * c2 + x <= L) ? __uint_as_float(r[0][x]) : 0.f;
                    rs1 += (j0 + 32 * c2 + 16 + x <= L) ? __uint_as_float(r[1][x]) : 0.f;
                }
            }
            float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
            for (int k = 0; k < CW / 8; ++k)
                qc[k] = *reinterpret_cast<const uint4 *>(st + ST_Q + (j0 >> 6) * SLAB +
                                                         sw128_offset(L, cs + 8 * k));
#pragma unroll
            for (int k = 0; k < CW / 8; ++k) {
                const uint32_t qw[4] = {qc[k].x, qc[k].y, qc[k].z, qc[k].w};
                const float4 ma = reinterpret_cast<const float4 *>(mb + j0)[2 * k];
                const float4 mc = reinterpret_cast<const float4 *>(mb + j0)[2 * k + 1];
                d0 = fmaf(ma.x, bf_lo(qw[0]), d0); d1 = fmaf(ma.y, bf_hi(qw[0]), d1);
                d2 = fmaf(ma.z, bf_lo(qw[1]), d2); d3 = fmaf(ma.w, bf_hi(qw[1]), d3);
                d0 = fmaf(mc.x, bf_lo(qw[2]), d0); d1 = fmaf(mc.y, bf_hi(qw[2]), d1);
                d2 = fmaf(mc.z, bf_lo(qw[3]), d2); d3 = fmaf(mc.w, bf_hi(qw[3]), d3);
            }
            fx[cg * NB + L] = (rs0 + rs1) + ((d0 + d1) + (d2 + d3));
            key_sums(st + ST_K);
            put_key_sums();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_empty[i % NST]);   // the stage is read
            // the q_clean store of block n - 2 has read its staging tile
            if (tid == 0) bulk_wait_group_read0();
            if (named_sync_or(1, NMAIN * 32, bad)) return true;
            const float nt = n0 + (float)(tok + 1);
            float xs = 0.f;
#pragma unroll
            for (int g = 0; g < NCG; ++g) xs += fx[g * NB + L];
            const float spn = xs / nt;
            {
                const float c = sum_key_sums();
                if (tid < 4 * D && (tid & 3) == 0) fm[((n + 1) % 3) * D + (tid >> 2)] = mb[tid >> 2] + c;
            }
            // ---- A'_n = G_ts - s_t for s <= t, else 0: bf16 pairs into TMEM
            const uint32_t tA = tb + lane_base + TM_A + 64u * (uint32_t)(n & 1) + (uint32_t)(j0 / 2);
#pragma unroll
            for (int h2 = 0; h2 < CW / 32; ++h2) {
                uint32_t w[16];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t r[16];
                    tmem_ld16(tb + lane_base + TM_G + j0 + 32 * h2 + 16 * c2, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s0 = j0 + 32 * h2 + 16 * c2 + 2 * e;
                        w[8 * c2 + e] = pack_bf2(s0 <= L ? __uint_as_float(r[2 * e]) - spn : 0.f,
                                                 s0 + 1 <= L ? __uint_as_float(r[2 * e + 1]) - spn : 0.f);
                    }
                }
                tmem_st16(tA + 16 * h2, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_a);
            if (n > 0) {
                // ---- block n - 1: finished from O_{n-1}; then M_n (Z_{n-1}
                //      added) to shared memory for O_n
                if (!__all_sync(0xffffffffu,
                                mbar_wait_or_abort(&bar_o, (uint32_t)((n - 1) & 1), &sAbort))) {
                    bad = true;
                    fail();
                }
                tc_fence_after();
                finish(n - 1, qp);
#pragma unroll
                for (int c4 = 0; c4 < CW / 16; ++c4) {
                    uint32_t r[16];
                    tmem_ld16(tM + 16 * c4, r);
                    tmem_ld_wait();
                    st_row16(sMs, L, cs + 16 * c4, r);
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_m);
            }
            sp = spn;
            scale = lam_n / nt;
            // the scratch rows (fx, fc) and m_{b+1} settle before the next block
            return named_sync_or(2, NMAIN * 32, bad);
        };

        uint4 qa[CW / 8], qb[CW / 8];
        bool stop = stop0;
        for (int n = 0; !stop && n < nb; n += 2) {
            if ((stop = step(n, qa, qb))) break;
            if (n + 1 < nb && (stop = step(n + 1, qb, qa))) break;
        }
        const bool aborted = named_sync_or(1, NMAIN * 32, bad || stop);
        if (!aborted) {
            if (!__all_sync(0xffffffffu,
                            mbar_wait_or_abort(&bar_o, (uint32_t)((nb - 1) & 1), &sAbort)))
                fail();
            tc_fence_after();
            if ((nb - 1) & 1) finish(nb - 1, qb); else finish(nb - 1, qa);
            if (seg == p.P - 1) {
                if (p.Ms_T) {
                    float *dst = p.Ms_T + ((size_t)unit * D + L) * D + j0;
                    const bool a16 = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
#pragma unroll
                    for (int c4 = 0; c4 < CW / 16; ++c4) {
                        uint32_t r[16];
                        tmem_ld16(tM + 16 * c4, r);
                        tmem_ld_wait();
                        if (a16) {
#pragma unroll
                            for (int x = 0; x < 4; ++x)
                                reinterpret_cast<float4 *>(dst + 16 * c4)[x] =
                                    make_float4(__uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                                                __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
                        } else {
#pragma unroll
                            for (int x = 0; x < 16; ++x) dst[16 * c4 + x] = __uint_as_float(r[x]);
                        }
                    }
                }
                if (p.ms_T && tid < D) p.ms_T[(size_t)unit * D + tid] = fm[(nb % 3) * D + tid];
                if (p.ns_T && tid == 0) p.ns_T[unit] = n0 + (float)p.T;
            }
        }
        if (tid == 0) bulk_wait_group0();   // the q_clean stores have completed
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

bool ccq_use_tc(int d, int dtype) { return chunk_tc_supported(d, dtype); }

int ccq_sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            return 148;
    }
    return n;
}

// Segments per (sequence, head): up to one CTA per SM, at most P_MAX.  A
// segment starting at block b0 with nb blocks costs PREFIX_COST b0 + nb; the
// cut minimises the largest cost (bisection on it, each segment as long as
// that cost allows).
struct CcqTcPlan {
    int P;
    int start[ctc::P_MAX + 1];
};
CcqTcPlan ccq_tc_plan(int B, int T, int H) {
    const int nblk = (T + ctc::NB - 1) / ctc::NB;
    const long units = std::max(1L, (long)B * H);
    const int Pmax = (int)std::max(1L, std::min({(long)ctc::P_MAX, ccq_sm_count() / units,
                                                 (long)nblk}));
    auto cut = [&](double c, CcqTcPlan &pl) {
        int b0 = 0, s = 0;
        pl.start[0] = 0;
        while (b0 < nblk && s < Pmax) {
            const int len = std::max(1, (int)(c - ctc::PREFIX_COST * b0 + 1e-9));
            b0 = std::min(nblk, b0 + len);
            pl.start[++s] = b0;
        }
        pl.P = s;
        return b0 >= nblk;
    };
    CcqTcPlan pl{};
    double lo = 0.0, hi = (double)nblk;
    for (int it = 0; it < 40; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (cut(mid, pl)) hi = mid; else lo = mid;
    }
    cut(hi, pl);
    return pl;
}

cudaError_t launch_ccq_tc(const CcqProblem &p, cudaStream_t s) {
    if (tmap::encode_fn() == nullptr) return cudaErrorNotSupported;
    const CcqTcPlan pl = ccq_tc_plan(p.B, p.T, p.H);
    const int units = p.B * p.H;
    CcqTcParams prm{};
    prm.lambda = p.lambda;
    prm.Ms0 = p.Ms0; prm.ms0 = p.ms0; prm.ns0 = p.ns0;
    prm.Ms_T = p.Ms_T; prm.ms_T = p.ms_T; prm.ns_T = p.ns_T;
    prm.status = static_cast<unsigned *>(p.ws);
    prm.T = p.T; prm.H = p.H; prm.P = pl.P;
    for (int i = 0; i <= pl.P; ++i) prm.seg_start[i] = pl.start[i];
    CUtensorMap mq, mk, mo;
    if (!tmap::seq_4d(&mq, p.q, p.B, p.T, p.H, ctc::NB) ||
        !tmap::seq_4d(&mk, p.k, p.B, p.T, p.H, ctc::NB) ||
        !tmap::seq_4d(&mo, p.q_clean, p.B, p.T, p.H, ctc::NB))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(p.ws, 0, sizeof(unsigned), s);   // status word
    if (e != cudaSuccess) return e;
    static bool attrs = false;
    if (!attrs) {
        if ((e = cudaFuncSetAttribute(ccq_query_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)ctc::SMEM)) != cudaSuccess)
            return e;
        attrs = true;
    }
    ccq_query_tc_kernel<<<units * pl.P, ctc::THREADS, ctc::SMEM, s>>>(mq, mk, mo, prm);
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
    if (ccq_use_tc(d, dtype)) return kWsHeader;   // the status word only
    const size_t nch = (size_t)(T + CC - 1) / CC;
    const size_t es = dtype == 1 ? 2 : 4;
    return kWsHeader + (size_t)B * H * nch * ((size_t)d * d * es + (size_t)d * 4);
}

cudaError_t launch_ccq(const CcqProblem &p, cudaStream_t s) {
    if (p.B == 0 || p.T == 0) return cudaSuccess;
    if (ccq_use_tc(p.d, p.dtype)) return launch_ccq_tc(p, s);
    if (p.dtype == 1)
        return p.d == 128 ? launch_ccq_t<__nv_bfloat16, 128>(p, s)
                          : launch_ccq_t<__nv_bfloat16, 64>(p, s);
    return p.d == 128 ? launch_ccq_t<float, 128>(p, s) : launch_ccq_t<float, 64>(p, s);
}

}  // namespace kla
