// Tensor-core (tcgen05 + TMEM + TMA) chunkwise KLA prefill: bf16 q/k/v,
// d = dk = dv = 128, chunk C = 64, fp32 state.
//
// Kaczmarz Linear Attention summary (gist.science 2605.08587), section
// "Implementacao": KLA keeps Gated DeltaNet's blockwise algorithm and only
// changes the diagonal coefficient matrix B = Diag(beta_1..beta_C) in the
// block solver; beta_t = eta_t / (||k_t||^2 + eps) (section "A Regra de
// Atualizacao KLA").  Per chunk (g = in-chunk cumulative log decay,
// Gamma_ts = exp(g_t - g_s)):
//
//   T  = (I + strict_lower(diag(beta) (Gamma o K K^T)))^{-1}
//   W  = T diag(beta) diag(exp g) K        U~ = T diag(beta) V
//   A  = lower(Gamma o Q K^T)
//   U  = U~ - W S
//   O  = diag(exp g) Q S + A U
//   S' = exp(g_C) S + K^T diag(exp(g_C - g)) U
//
// Phase 1 (intra_kernel) is parallel over every (chunk, head): two chunks per
// CTA so that every tensor-core product has M = 128 rows.  It computes
// K K^T and Q K^T on tcgen05 (TMEM accumulators), solves T in fp32 by
// forward substitution (one column per thread, registers), and forms
// [W | U~] = (T diag(beta)) [diag(exp g) K | V] with a single N = 256 MMA.
// W, U~, A (bf16) and g (fp32) go to the caller's workspace.
//
// Phase 2 (state_kernel) walks the chunks of one (sequence, head) in order.
// It works on transposed products so that M = dv = 128:
//   P^T  = S^T W^T           (A = S^T bf16 in smem, B = W tile)
//   X^T  = S^T Q^T
//   U^T  = U~^T - P^T        (registers -> bf16 smem tile)
//   Y^T  = U^T A^T
//   Z^T  = (U diag(exp(g_C - g)))^T K
//   O^T  = X^T diag(exp g) + Y^T ;  S^T <- exp(g_C) S^T + Z^T (fp32 in registers)
// Its next chunk's tiles stream in by TMA while the current chunk computes.
//
// All waits are bounded (kla_tc.cuh); a wait that gives up sets the status
// word to a timeout code and the CTA leaves after releasing TMEM.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "kla_internal.h"
#include "kla_tc.cuh"

namespace kla {
namespace {

using namespace tc;

constexpr int D = 128;     // dk = dv
constexpr int C = kChunk;  // 64

struct TcParams {
    int H, n_seq, T, nch_fixed;
    int total_T;
    float eps;
    const float *alpha, *eta, *S0;
    float *S_T;
    __nv_bfloat16 *o;
    const int *cu_seqlens;     // varlen only
    const int *chunk_prefix;   // varlen only: first chunk of each sequence, [N+1]
    const int *order;          // varlen only: sequences by decreasing length, [N]
    unsigned *status;
    float *g_ws;               // [slots][64]
    __nv_bfloat16 *W_ws;       // [slots][64][128]
    __nv_bfloat16 *U_ws;       // [slots][64][128]
    __nv_bfloat16 *A_ws;       // [slots][64][64]
};

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
    const uint32_t a = smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ void set_status(unsigned *status, unsigned code) {
    if (status) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ bool status_bad(const unsigned *status) {
    return status != nullptr && *(volatile const unsigned *)status != kDevOk;
}

// Chunk g of head h: its sequence, first token row, valid length.  False when
// g lies beyond the last chunk (the grid is sized by an upper bound).
__device__ __forceinline__ bool slot_info(const TcParams &p, long g, int &seq, long &row0,
                                          int &nc) {
    if (p.chunk_prefix == nullptr) {
        if (p.nch_fixed <= 0) return false;
        seq = (int)(g / p.nch_fixed);
        if (seq >= p.n_seq) return false;
        const int c = (int)(g % p.nch_fixed);
        row0 = (long)seq * p.T + (long)c * C;
        nc = min(C, p.T - c * C);
        return true;
    }
    const int total = p.chunk_prefix[p.n_seq];
    if (g >= total) return false;
    int lo = 0, hi = p.n_seq - 1;  // last sequence whose first chunk is <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.chunk_prefix[mid] <= g) lo = mid; else hi = mid - 1;
    }
    seq = lo;
    const int c = (int)(g - p.chunk_prefix[seq]);
    const long start = p.cu_seqlens[seq];
    const long len = (long)p.cu_seqlens[seq + 1] - start;
    row0 = start + (long)c * C;
    nc = (int)min((long)C, len - (long)c * C);
    return nc > 0;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // a -> low half
    return *reinterpret_cast<const uint32_t *>(&v);
}

// ===================================================================== phase 1
constexpr int P1_THREADS = 128;
constexpr uint32_t P1_SMEM = 3 * 32768 + 1024;  // K, V, Q/L/A regions + alignment slack

__global__ void __launch_bounds__(P1_THREADS, 2)
intra_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mv, const TcParams p) {
    extern __shared__ unsigned char smraw[];
    __shared__ uint64_t bars[3];
    __shared__ uint32_t tslot;
    __shared__ float sG[128], sBeta[128], sCarry[4];
    __shared__ int sAbort;

    unsigned char *sm = align1024(smraw);
    unsigned char *sK = sm;           // [2 slabs][128 rows][128 B]; later diag(exp g) K
    unsigned char *sV = sm + 32768;   // same layout (n-block stride 16 KB continues from sK)
    unsigned char *sQ = sm + 65536;   // Q tile -> fp32 L[2][64][64] -> A operand T diag(beta)
    float *sL = reinterpret_cast<float *>(sQ);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    if (status_bad(p.status)) return;

    int seqs[2], ncs[2];
    long row0s[2];
    bool valid[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        valid[q] = slot_info(p, 2L * blockIdx.x + q, seqs[q], row0s[q], ncs[q]);
        if (!valid[q]) { ncs[q] = 0; row0s[q] = 0; }
    }
    if (!valid[0] && !valid[1]) return;

    const int slot = tid >> 6, t = tid & 63;
    const int nc = ncs[slot];

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_mbar_init();
        sAbort = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 256);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tslot;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    if (tid == 0) {
        tma_prefetch_map(&mk);
        mbar_expect_tx(&bars[0], 3u * 32768u);
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int z = (int)row0s[q];
                tma_load_3d(sK + s * 16384 + q * 8192, &mk, &bars[0], 64 * s, h, z);
                tma_load_3d(sQ + s * 16384 + q * 8192, &mq, &bars[0], 64 * s, h, z);
                tma_load_3d(sV + s * 16384 + q * 8192, &mv, &bars[0], 64 * s, h, z);
            }
    }

    // ---- decay: g = inclusive prefix sum of log alpha within each chunk ----
    float a = 1.f, et = 0.f;
    if (t < nc) {
        const size_t row = (size_t)(row0s[slot] + t) * p.H + h;
        a = p.alpha[row];
        et = p.eta[row];
    }
    double gs = (double)logf(a);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double u = __shfl_up_sync(0xffffffffu, gs, off);
        if (lane >= off) gs += u;
    }
    if (lane == 31) sCarry[warp] = (float)gs;
    __syncthreads();
    if (warp & 1) gs += (double)sCarry[warp - 1];
    sG[tid] = (float)gs;

    // ---- tiles landed: Gram products on the tensor cores ----
    if (!mbar_wait(&bars[0], 0)) {
        sAbort = 1;
        set_status(p.status, kDevTimeout);
    }
    __syncthreads();
    const bool abort1 = sAbort != 0;
    if (tid == 0 && !abort1) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
        const uint32_t aK = smem_u32(sK), aQ = smem_u32(sQ);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            mma_bf16(tb + 0, sdesc_sw128(aK + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024),
                     idesc, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            mma_bf16(tb + 128, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024),
                     idesc, ks > 0);
        }
        mma_commit(&bars[1]);
    }

    // ---- beta_t from the key's squared norm (fp32 over the bf16 values) ----
    {
        float n2 = 0.f;
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint4 v = *reinterpret_cast<const uint4 *>(sK + s * 16384 +
                                                                sw128_offset(tid, ch * 8));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float x0 = bf_lo(w[i]), x1 = bf_hi(w[i]);
                    n2 = fmaf(x0, x0, n2);
                    n2 = fmaf(x1, x1, n2);
                }
            }
        const float den = n2 + p.eps;
        sBeta[tid] = (t < nc && den != 0.f) ? et / den : 0.f;
    }
    __syncthreads();

    // ---- epilogue 1: L = strict_lower(beta Gamma o KK^T) (fp32 smem), A = lower(Gamma o QK^T) ----
    bool ok = !abort1 && mbar_wait(&bars[1], 0);
    if (!abort1 && !ok) set_status(p.status, kDevTimeout);
    tc_fence_after();
    const float gt = sG[tid];
    const float bt = sBeta[tid];
    const int cb = slot * 64;
    const long gidx0 = 2L * blockIdx.x + slot;
    const size_t slot_row = (size_t)(gidx0 * p.H + h) * C + t;   // row of this token in the ws
    if (ok) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            tmem_ld32(tb + lane_base + cb + half * 32, r);
            tmem_ld_wait();
            float *Lrow = sL + (size_t)(slot * 64 + t) * 64 + half * 32;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int s = half * 32 + i;
                const float gam = (s < t) ? __expf(gt - sG[cb + s]) : 0.f;
                Lrow[i] = (s < t && t < nc) ? bt * gam * __uint_as_float(r[i]) : 0.f;
            }
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            tmem_ld32(tb + lane_base + 128 + cb + half * 32, r);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const int s = half * 32 + i;
                const float a0 = (s <= t && t < nc)
                                     ? __expf(gt - sG[cb + s]) * __uint_as_float(r[i]) : 0.f;
                const float a1 = (s + 1 <= t && t < nc)
                                     ? __expf(gt - sG[cb + s + 1]) * __uint_as_float(r[i + 1]) : 0.f;
                pk[i / 2] = pack_bf2(a0, a1);
            }
            if (valid[slot]) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.A_ws + slot_row * 64 + half * 32);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
        }
        // K row -> diag(exp g) K; rows past the chunk's end (another
        // sequence's tokens or TMA zero fill) are cleared in K and V so that
        // nothing from them can reach the products.
        const float gam_t = __expf(gt);
        const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 *pk4 = reinterpret_cast<uint4 *>(sK + s * 16384 + sw128_offset(tid, ch * 8));
                if (t < nc) {
                    const uint4 v = *pk4;
                    *pk4 = make_uint4(pack_bf2(gam_t * bf_lo(v.x), gam_t * bf_hi(v.x)),
                                      pack_bf2(gam_t * bf_lo(v.y), gam_t * bf_hi(v.y)),
                                      pack_bf2(gam_t * bf_lo(v.z), gam_t * bf_hi(v.z)),
                                      pack_bf2(gam_t * bf_lo(v.w), gam_t * bf_hi(v.w)));
                } else {
                    *pk4 = zero4;
                    *reinterpret_cast<uint4 *>(sV + s * 16384 + sw128_offset(tid, ch * 8)) = zero4;
                }
            }
    }
    if (!ok) sAbort = 1;
    __syncthreads();
    const bool abort2 = sAbort != 0;

    // ---- T = (I + L)^{-1}: this thread solves column j = t of its chunk ----
    float x[64];
    {
        const float *Lb = sL + (size_t)slot * 64 * 64;
#pragma unroll
        for (int tt = 0; tt < 64; ++tt) {
            float acc = (tt == t) ? 1.f : 0.f;
            const float *Lrow = Lb + tt * 64;
#pragma unroll
            for (int s = 0; s < tt; ++s) acc = fmaf(-Lrow[s], x[s], acc);
            x[tt] = acc;
        }
    }
    __syncthreads();  // every thread is done with L; its region becomes the A operand

    // ---- A operand = T diag(beta), block diagonal over the two chunks ----
    {
        const float bj = sBeta[tid];
        unsigned char *slab = sQ + slot * 16384;   // columns of this chunk
#pragma unroll
        for (int rr = 0; rr < 128; ++rr) {
            const float val = ((rr >> 6) == slot) ? x[rr & 63] * bj : 0.f;
            *reinterpret_cast<__nv_bfloat16 *>(slab + sw128_offset(rr, t)) = __float2bfloat16_rn(val);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && !abort2) {
        tc_fence_after();
        // [W | U~] = (T diag beta) [diag(exp g) K | V]: M=128, N=256, K=128 tokens.
        // B is MN-major (rows = tokens): n-blocks of 64 at 16 KB stride
        // (sK slab 0, sK slab 1, sV slab 0, sV slab 1).
        const uint32_t idesc = idesc_bf16_f32(128, 256, false, true);
        const uint32_t aA = smem_u32(sQ), aB = smem_u32(sK);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint64_t da = sdesc_sw128(aA + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
            const uint64_t db = sdesc_sw128(aB + ks * 2048, 16384, 1024);
            mma_bf16(tb + 0, da, db, idesc, ks > 0);
        }
        mma_commit(&bars[2]);
    }
    __syncthreads();

    // ---- epilogue 2: W, U~ rows (bf16) and g to the workspace ----
    ok = !abort2 && mbar_wait(&bars[2], 0);
    if (!abort2 && !ok) set_status(p.status, kDevTimeout);
    tc_fence_after();
    if (ok && valid[slot]) {
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            __nv_bfloat16 *dst_row = (part == 0 ? p.W_ws : p.U_ws) + slot_row * D;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t r[32];
                tmem_ld32(tb + lane_base + part * 128 + c4 * 32, r);
                tmem_ld_wait();
                uint4 *dst = reinterpret_cast<uint4 *>(dst_row + c4 * 32);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    dst[v4] = make_uint4(
                        pack_bf2(__uint_as_float(r[8 * v4 + 0]), __uint_as_float(r[8 * v4 + 1])),
                        pack_bf2(__uint_as_float(r[8 * v4 + 2]), __uint_as_float(r[8 * v4 + 3])),
                        pack_bf2(__uint_as_float(r[8 * v4 + 4]), __uint_as_float(r[8 * v4 + 5])),
                        pack_bf2(__uint_as_float(r[8 * v4 + 6]), __uint_as_float(r[8 * v4 + 7])));
            }
        }
        p.g_ws[slot_row] = gt;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 256);
}

// ===================================================================== phase 2
constexpr int P2_THREADS = 256;
constexpr uint32_t ST_W = 0, ST_Q = 16384, ST_K = 32768, ST_U = 49152, ST_A = 65536,
                   ST_G = 73728, ST_BYTES = 74752;   // stage layout (1 KB aligned pieces)
constexpr uint32_t ST_TX = 16384u * 4u + 8192u + 256u;  // bytes a stage receives
constexpr uint32_t P2_OFF_S = 2 * ST_BYTES;             // S^T bf16 [128][128] (2 slabs)
constexpr uint32_t P2_OFF_UT = P2_OFF_S + 32768;        // U^T bf16 [128][64]
constexpr uint32_t P2_OFF_US = P2_OFF_UT + 16384;       // (U diag(exp(gC-g)))^T [128][64]
constexpr uint32_t P2_SMEM = P2_OFF_US + 16384 + 1024;

// TMEM columns (fp32): P^T 0..63, X^T 64..127, Y^T 128..191, Z^T 256..383.
constexpr uint32_t TM_P = 0, TM_X = 64, TM_Y = 128, TM_Z = 256;

__device__ __forceinline__ void issue_stage(unsigned char *st, uint64_t *bar,
                                            const CUtensorMap *mq, const CUtensorMap *mk,
                                            const CUtensorMap *mw, const CUtensorMap *mu,
                                            const CUtensorMap *ma, const float *g_src, int h,
                                            int row0, int slot) {
    mbar_expect_tx(bar, ST_TX);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        tma_load_2d(st + ST_W + s * 8192, mw, bar, 64 * s, slot * C);
        tma_load_3d(st + ST_Q + s * 8192, mq, bar, 64 * s, h, row0);
        tma_load_3d(st + ST_K + s * 8192, mk, bar, 64 * s, h, row0);
        tma_load_2d(st + ST_U + s * 8192, mu, bar, 64 * s, slot * C);
    }
    tma_load_2d(st + ST_A, ma, bar, 0, slot * C);
    bulk_load(st + ST_G, g_src, 256, bar);
}

__global__ void __launch_bounds__(P2_THREADS, 1)
state_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
             const __grid_constant__ CUtensorMap ma, const TcParams p) {
    extern __shared__ unsigned char smraw[];
    __shared__ uint64_t bar_ld[2];
    __shared__ uint64_t bar_p, bar_s;
    __shared__ uint32_t tslot;
    __shared__ int sAbort;

    unsigned char *sm = align1024(smraw);
    unsigned char *sS = sm + P2_OFF_S;
    unsigned char *sUt = sm + P2_OFF_UT;
    unsigned char *sUs = sm + P2_OFF_US;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int j = quarter * 32 + lane;          // dv index = TMEM lane of this thread
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;

    if (status_bad(p.status)) return;
    const int rank = blockIdx.x / p.H, h = blockIdx.x % p.H;
    const int seq = p.order ? p.order[rank] : rank;
    long start, len, chunk0;
    if (p.cu_seqlens) {
        start = p.cu_seqlens[seq];
        len = (long)p.cu_seqlens[seq + 1] - start;
        chunk0 = p.chunk_prefix[seq];
    } else {
        start = (long)seq * p.T;
        len = p.T;
        chunk0 = (long)seq * p.nch_fixed;
    }
    const int nch = (int)((len + C - 1) / C);
    const size_t sbase = ((size_t)seq * p.H + h) * D * D;

    if (tid == 0) {
        mbar_init(&bar_ld[0], 1);
        mbar_init(&bar_ld[1], 1);
        mbar_init(&bar_p, 1);
        mbar_init(&bar_s, 1);
        fence_mbar_init();
        sAbort = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 512);
        tmem_relinquish();
    }

    // fp32 master state: this thread keeps S[i][j] for i in [64*half, 64*half+64)
    float Sr[64];
#pragma unroll
    for (int i = 0; i < 64; ++i)
        Sr[i] = p.S0 ? p.S0[sbase + (size_t)(64 * half + i) * D + j] : 0.f;
    // bf16 copy as the A operand S^T (row j, K-major, slab = half)
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4 *>(sS + half * 16384 + sw128_offset(j, ch * 8)) =
            make_uint4(pack_bf2(Sr[8 * ch + 0], Sr[8 * ch + 1]), pack_bf2(Sr[8 * ch + 2], Sr[8 * ch + 3]),
                       pack_bf2(Sr[8 * ch + 4], Sr[8 * ch + 5]), pack_bf2(Sr[8 * ch + 6], Sr[8 * ch + 7]));
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tslot;

    if (tid == 0) {
        for (int c = 0; c < 2 && c < nch; ++c) {
            const long slot = (chunk0 + c) * p.H + h;
            issue_stage(sm + c * ST_BYTES, &bar_ld[c], &mq, &mk, &mw, &mu, &ma,
                        p.g_ws + slot * C, h, (int)(start + (long)c * C), (int)slot);
        }
    }

    const uint32_t id_n64 = idesc_bf16_f32(128, 64, false, false);
    const uint32_t id_z = idesc_bf16_f32(128, 128, false, true);
    bool abort = false;
    for (int c = 0; c < nch; ++c) {
        const int b = c & 1;
        unsigned char *st = sm + b * ST_BYTES;
        const uint32_t par_ld = (uint32_t)((c >> 1) & 1);
        const uint32_t par = (uint32_t)(c & 1);
        const int nc = (int)min((long)C, len - (long)c * C);
        const long row0 = start + (long)c * C;

        // ---- P^T = S^T W^T and X^T = S^T Q^T ----
        if (tid == 0) {
            if (!mbar_wait(&bar_ld[b], par_ld)) {
                sAbort = 1;
                set_status(p.status, kDevTimeout);
            } else {
                tc_fence_after();
                const uint32_t aS = smem_u32(sS), aW = smem_u32(st + ST_W), aQ = smem_u32(st + ST_Q);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
                    const uint32_t offS = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tb + TM_P, sdesc_sw128(aS + offS, 16, 1024),
                             sdesc_sw128(aW + off, 16, 1024), id_n64, ks > 0);
                }
                mma_commit(&bar_p);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
                    const uint32_t offS = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tb + TM_X, sdesc_sw128(aS + offS, 16, 1024),
                             sdesc_sw128(aQ + off, 16, 1024), id_n64, ks > 0);
                }
            }
        }
        // every thread needs the stage's g and U~ as well
        const bool landed = mbar_wait(&bar_ld[b], par_ld);
        if (landed && nc < C) {
            // partial chunk: clear K rows past its end (read only by the
            // state-update product, issued after the next barrier)
            for (int x = tid; x < (C - nc) * 16; x += P2_THREADS) {
                const int row = nc + (x >> 4), sl = (x >> 3) & 1, ch = x & 7;
                *reinterpret_cast<uint4 *>(st + ST_K + sl * 8192 + sw128_offset(row, ch * 8)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (!landed || !mbar_wait(&bar_p, par)) {
            set_status(p.status, kDevTimeout);
            sAbort = 1;
        }
        __syncthreads();
        if (sAbort) { abort = true; break; }
        tc_fence_after();

        // ---- U^T = U~^T - P^T for tokens [32*half, 32*half + 32) ----
        const float *gch = reinterpret_cast<const float *>(st + ST_G);
        const float gC = gch[C - 1];
        {
            uint32_t r[32];
            tmem_ld32(tb + lane_base + TM_P + half * 32, r);
            tmem_ld_wait();
            const unsigned char *sU = st + ST_U + (j >> 6) * 8192;
            uint32_t pu[16], ps[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const int t0 = half * 32 + i;
                const float u0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                     sU + sw128_offset(t0, j & 63))) - __uint_as_float(r[i]);
                const float u1 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                     sU + sw128_offset(t0 + 1, j & 63))) - __uint_as_float(r[i + 1]);
                pu[i / 2] = pack_bf2(u0, u1);
                ps[i / 2] = pack_bf2(u0 * __expf(gC - gch[t0]), u1 * __expf(gC - gch[t0 + 1]));
            }
            // row j of the [128][64] K-major tiles, columns 32*half.. (4 x 16 B)
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
                const uint32_t off = sw128_offset(j, half * 32 + v4 * 8);
                *reinterpret_cast<uint4 *>(sUt + off) =
                    make_uint4(pu[4 * v4], pu[4 * v4 + 1], pu[4 * v4 + 2], pu[4 * v4 + 3]);
                *reinterpret_cast<uint4 *>(sUs + off) =
                    make_uint4(ps[4 * v4], ps[4 * v4 + 1], ps[4 * v4 + 2], ps[4 * v4 + 3]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- Y^T = U^T A^T and Z^T = (U diag(exp(gC-g)))^T K ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t aUt = smem_u32(sUt), aUs = smem_u32(sUs);
            const uint32_t aA = smem_u32(st + ST_A), aK = smem_u32(st + ST_K);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tb + TM_Y, sdesc_sw128(aUt + ks * 32, 16, 1024),
                         sdesc_sw128(aA + ks * 32, 16, 1024), id_n64, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tb + TM_Z, sdesc_sw128(aUs + ks * 32, 16, 1024),
                         sdesc_sw128(aK + ks * 2048, 8192, 1024), id_z, ks > 0);
            mma_commit(&bar_s);
        }
        if (!mbar_wait(&bar_s, par)) {
            set_status(p.status, kDevTimeout);
            sAbort = 1;
        }
        tc_fence_after();

        // ---- S^T <- exp(gC) S^T + Z^T ; new bf16 copy of S^T ----
        if (!sAbort) {
            const float egC = __expf(gC);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r[32];
                tmem_ld32(tb + lane_base + TM_Z + half * 64 + c2 * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    Sr[c2 * 32 + i] = fmaf(egC, Sr[c2 * 32 + i], __uint_as_float(r[i]));
            }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4 *>(sS + half * 16384 + sw128_offset(j, ch * 8)) =
                    make_uint4(pack_bf2(Sr[8 * ch + 0], Sr[8 * ch + 1]),
                               pack_bf2(Sr[8 * ch + 2], Sr[8 * ch + 3]),
                               pack_bf2(Sr[8 * ch + 4], Sr[8 * ch + 5]),
                               pack_bf2(Sr[8 * ch + 6], Sr[8 * ch + 7]));

            // ---- O^T = X^T diag(exp g) + Y^T -> o[t][j] ----
            uint32_t rx[32], ry[32];
            tmem_ld32(tb + lane_base + TM_X + half * 32, rx);
            tmem_ld32(tb + lane_base + TM_Y + half * 32, ry);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int t = half * 32 + i;
                if (t < nc) {
                    const float ov = fmaf(__expf(gch[t]), __uint_as_float(rx[i]), __uint_as_float(ry[i]));
                    p.o[((size_t)(row0 + t) * p.H + h) * D + j] = __float2bfloat16_rn(ov);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (sAbort) { abort = true; break; }

        // ---- refill this stage with chunk c + 2 ----
        if (tid == 0 && c + 2 < nch) {
            const long slot = (chunk0 + c + 2) * p.H + h;
            issue_stage(st, &bar_ld[b], &mq, &mk, &mw, &mu, &ma, p.g_ws + slot * C, h,
                        (int)(start + (long)(c + 2) * C), (int)slot);
        }
    }

    if (!abort && p.S_T) {
#pragma unroll
        for (int i = 0; i < 64; ++i) p.S_T[sbase + (size_t)(64 * half + i) * D + j] = Sr[i];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// ===================================================================== varlen prep
// One CTA: validates cu_seqlens, writes the first chunk of every sequence
// (chunk_prefix[N+1]) and a longest-first order of the sequences.
constexpr int PREP_THREADS = 1024;

__global__ void __launch_bounds__(PREP_THREADS)
prep_kernel(const int *cu, int N, int total_T, int *chunk_prefix, int *order, unsigned *status) {
    __shared__ int bad;
    __shared__ int warp_sums[PREP_THREADS / 32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        bad = (cu[0] != 0 || cu[N] != total_T) ? 1 : 0;
        carry = 0;
    }
    __syncthreads();
    for (int i = tid; i < N; i += PREP_THREADS)
        if (cu[i + 1] < cu[i]) atomicOr(&bad, 1);
    __syncthreads();
    if (bad) {
        if (tid == 0) *status = kDevBadSeqlens;
        return;
    }
    for (int base = 0; base < N; base += PREP_THREADS) {
        const int i = base + tid;
        const int v = (i < N) ? (cu[i + 1] - cu[i] + C - 1) / C : 0;
        int x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += u;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += u;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
        if (i < N) chunk_prefix[i] = incl - v;
        __syncthreads();
        if (tid == PREP_THREADS - 1) carry = incl;
        __syncthreads();
    }
    if (tid == 0) chunk_prefix[N] = carry;
    // longest-first order (stable); identity for very large N
    for (int n = tid; n < N; n += PREP_THREADS) {
        int rank = n;
        if (N <= 8192) {
            const int ln = cu[n + 1] - cu[n];
            rank = 0;
            for (int m = 0; m < N; ++m) {
                const int lm = cu[m + 1] - cu[m];
                rank += (lm > ln) || (lm == ln && m < n);
            }
        }
        order[rank] = n;
    }
    if (tid == 0) *status = kDevOk;
}

// ===================================================================== host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool map_3d_rows(CUtensorMap *m, const void *base, int H, long rows) {
    // [rows][H][128] bf16; box = 64 feature columns x 1 head x 64 rows
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
    const cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                       strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool map_2d(CUtensorMap *m, const void *base, int cols, long rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)C};
    const cuuint32_t es[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                       strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
    size_t meta, g, W, U, A, total;
};

WsLayout layout(long n_chunks, int H, int n_seq) {
    const size_t slots = (size_t)n_chunks * H;
    WsLayout L;
    L.meta = 0;
    L.g = align_up(((size_t)2 * n_seq + 1) * sizeof(int), 1024);
    L.W = L.g + align_up(slots * C * sizeof(float), 1024);
    L.U = L.W + slots * C * D * 2;
    L.A = L.U + slots * C * D * 2;
    L.total = L.A + slots * C * C * 2;
    return L;
}

}  // namespace

bool chunk_tc_supported(int d, int dtype) { return d == 128 && dtype == 1; }

size_t chunk_tc_workspace_bytes(long n_chunks_upper, int H, int n_seq) {
    return layout(n_chunks_upper, H, n_seq).total;
}

cudaError_t launch_chunk_tc(const Problem &p, long n_chunks_upper, cudaStream_t s) {
    if (p.n_seq == 0) return cudaSuccess;
    if (encode_fn() == nullptr) return cudaErrorNotSupported;
    const WsLayout L = layout(n_chunks_upper, p.H, p.n_seq);
    unsigned char *ws = static_cast<unsigned char *>(p.ws);
    if (p.ws_bytes < L.total) return cudaErrorInvalidValue;

    TcParams tp{};
    tp.H = p.H;
    tp.n_seq = p.n_seq;
    tp.T = p.T;
    tp.total_T = p.total_T;
    tp.nch_fixed = p.cu_seqlens ? 0 : (p.T + C - 1) / C;
    tp.eps = p.eps;
    tp.alpha = p.alpha;
    tp.eta = p.eta;
    tp.S0 = p.S0;
    tp.S_T = p.S_T;
    tp.o = static_cast<__nv_bfloat16 *>(p.o);
    tp.cu_seqlens = p.cu_seqlens;
    tp.status = p.status;
    tp.g_ws = reinterpret_cast<float *>(ws + L.g);
    tp.W_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.W);
    tp.U_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.U);
    tp.A_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.A);
    int *chunk_prefix = reinterpret_cast<int *>(ws + L.meta);
    int *order = chunk_prefix + p.n_seq + 1;
    tp.chunk_prefix = p.cu_seqlens ? chunk_prefix : nullptr;
    tp.order = p.cu_seqlens ? order : nullptr;

    CUtensorMap mq, mk, mv, mw, mu, ma;
    const long slots = n_chunks_upper * p.H;
    if (!map_3d_rows(&mq, p.q, p.H, p.total_T) || !map_3d_rows(&mk, p.k, p.H, p.total_T) ||
        !map_3d_rows(&mv, p.v, p.H, p.total_T) || !map_2d(&mw, tp.W_ws, D, slots * C) ||
        !map_2d(&mu, tp.U_ws, D, slots * C) || !map_2d(&ma, tp.A_ws, C, slots * C))
        return cudaErrorInvalidValue;

    cudaError_t e;
    if (p.cu_seqlens) {
        prep_kernel<<<1, PREP_THREADS, 0, s>>>(p.cu_seqlens, p.n_seq, p.total_T, chunk_prefix,
                                               order, p.status);
        note_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    static bool attrs = false;
    if (!attrs) {
        if ((e = cudaFuncSetAttribute(intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)P1_SMEM)) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)P2_SMEM)) != cudaSuccess)
            return e;
        attrs = true;
    }
    dim3 g1((unsigned)((n_chunks_upper + 1) / 2), (unsigned)p.H);
    intra_kernel<<<g1, P1_THREADS, P1_SMEM, s>>>(mq, mk, mv, tp);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    state_kernel<<<(unsigned)(p.n_seq * p.H), P2_THREADS, P2_SMEM, s>>>(mq, mk, mw, mu, ma, tp);
    note_launch();
    return cudaGetLastError();
}

}  // namespace kla
