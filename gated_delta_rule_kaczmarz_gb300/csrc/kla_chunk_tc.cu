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
// work item so that every tensor-core product has M = 128 rows; CTAs are
// persistent.  It computes K K^T and Q K^T on tcgen05 (TMEM accumulators),
// inverts I + L in fp32 on the CUDA cores (forward substitution on 16 x 16
// diagonal blocks, then two doubling steps made of small products), and forms
// W = (T diag beta)(diag(exp g) K) and U~^T = V^T (T diag beta)^T with two
// MMAs.  W, U~^T, A^T and diag(exp(g_C - g)) K (bf16) and exp(g) (fp32) go to
// the caller's workspace.
//
// Phase 2 (state_kernel) walks the chunks of one (sequence, head) in order,
// every product with M = dv = 128 rows and the two products of a step fused
// into one wide MMA (issue cost per tcgen05.mma is nearly independent of N):
//   [P^T | X^T] = S^T [W ; Q]^T ;  U^T = U~^T - P^T
//   [Z^T | Y^T] = U^T [diag(exp(g_C - g)) K | A^T]
//   S^T <- exp(g_C) S^T + Z^T (fp32 registers) ;  O^T = X^T diag(exp g) + Y^T
// The serial chain is P -> U -> Z -> S; a dedicated warp issues the MMAs and
// TMA loads (three chunks in flight), and the chain's warps store a chunk's
// outputs while the next chunk's first product runs.  S^T and U^T, the bf16 A
// operands, are kept in tensor memory.
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
    float *eg_ws;              // [slots][64]        exp(g_t)
    __nv_bfloat16 *Kt_ws;      // [slots][64][128]   diag(exp(g_C - g)) K
    __nv_bfloat16 *W_ws;       // [slots][64][128]
    __nv_bfloat16 *UT_ws;      // [slots][128][64]  U~ transposed (feature-major)
    __nv_bfloat16 *A_ws;       // [slots][64 keys s][64 queries t]  A^T
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

// Packs 32 fp32 values (as raw bits) to bf16 and stores them (64 bytes).
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16 *dst, const uint32_t (&r)[32]) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4)
        d4[v4] = make_uint4(
            pack_bf2(__uint_as_float(r[8 * v4 + 0]), __uint_as_float(r[8 * v4 + 1])),
            pack_bf2(__uint_as_float(r[8 * v4 + 2]), __uint_as_float(r[8 * v4 + 3])),
            pack_bf2(__uint_as_float(r[8 * v4 + 4]), __uint_as_float(r[8 * v4 + 5])),
            pack_bf2(__uint_as_float(r[8 * v4 + 6]), __uint_as_float(r[8 * v4 + 7])));
}

// fp32 64 x 64 matrices in shared memory, one per chunk, rows of 64 floats;
// the float4 index within a row is XORed with (row % 16) so that a thread per
// row writing float4s, and a warp reading one row as a broadcast, are both
// free of bank conflicts.  Offset of (row, col) within the matrix rows:
__device__ __forceinline__ int lsw(int row, int col) {
    return ((((col >> 2) ^ (row & 15))) << 2) | (col & 3);
}

// fp32 64 x 64 matrix of chunk p (L, then T) in phase 1: it occupies the
// 16 KB that chunk p's half of the Q tile used, in 64-feature slab p.
__device__ __forceinline__ float *lslot(unsigned char *kq, int p) {
    return reinterpret_cast<float *>(kq + p * 32768 + 16384);
}

// One doubling step of the blocked inverse, in place in the fp32 L storage
// of both chunks: for every diagonal block of size 2n whose two diagonal
// n x n blocks already hold D1 = (I + L11)^{-1} and D2 = (I + L22)^{-1},
// replace its lower-left block L21 by -D2 L21 D1.  128 threads; each computes
// an (n/8) x 4 patch of the n x n products.
template <int n>
__device__ __forceinline__ void merge_level(unsigned char *kq, int tid) {
    constexpr int nblk = 64 / (2 * n);               // blocks of size 2n per chunk
    constexpr int tpb = 128 / (2 * nblk);            // threads per block (both chunks)
    constexpr int rows = n * n / 4 / tpb;            // patch rows per thread (4 columns each)
    static_assert(rows * 4 * tpb == n * n, "patch tiling");
    const int blkid = tid / tpb, q = tid % tpb;
    const int p = blkid / nblk, o = 2 * n * (blkid % nblk);
    constexpr int pcols = n / 4;                     // column patches per row band
    const int pr = q / pcols, pc = q % pcols;        // rows [rows*pr, +rows), cols [4pc, +4)
    float *Lp = lslot(kq, p);
    float acc[rows][4];
    // M = L21 D1
#pragma unroll
    for (int m = 0; m < rows; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
#pragma unroll 2
    for (int s4 = 0; s4 < n / 4; ++s4) {
        float4 bb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = o + 4 * s4 + e;
            bb[e] = *reinterpret_cast<const float4 *>(Lp + r * 64 + lsw(r, o + 4 * pc));
        }
#pragma unroll
        for (int m = 0; m < rows; ++m) {
            const int r = o + n + rows * pr + m;
            const float4 a = *reinterpret_cast<const float4 *>(Lp + r * 64 + lsw(r, o + 4 * s4));
            const float am[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[m][0] = fmaf(am[e], bb[e].x, acc[m][0]);
                acc[m][1] = fmaf(am[e], bb[e].y, acc[m][1]);
                acc[m][2] = fmaf(am[e], bb[e].z, acc[m][2]);
                acc[m][3] = fmaf(am[e], bb[e].w, acc[m][3]);
            }
        }
    }
    __syncthreads();  // L21 fully read
#pragma unroll
    for (int m = 0; m < rows; ++m) {
        const int r = o + n + rows * pr + m;
        *reinterpret_cast<float4 *>(Lp + r * 64 + lsw(r, o + 4 * pc)) =
            make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
        acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
    }
    __syncthreads();  // M stored where L21 was
    // X = -D2 M
#pragma unroll 2
    for (int s4 = 0; s4 < n / 4; ++s4) {
        float4 bb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = o + n + 4 * s4 + e;
            bb[e] = *reinterpret_cast<const float4 *>(Lp + r * 64 + lsw(r, o + 4 * pc));
        }
#pragma unroll
        for (int m = 0; m < rows; ++m) {
            const int r = o + n + rows * pr + m;
            const float4 a = *reinterpret_cast<const float4 *>(Lp + r * 64 + lsw(r, o + n + 4 * s4));
            const float am[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[m][0] = fmaf(am[e], bb[e].x, acc[m][0]);
                acc[m][1] = fmaf(am[e], bb[e].y, acc[m][1]);
                acc[m][2] = fmaf(am[e], bb[e].z, acc[m][2]);
                acc[m][3] = fmaf(am[e], bb[e].w, acc[m][3]);
            }
        }
    }
    __syncthreads();  // M fully read
#pragma unroll
    for (int m = 0; m < rows; ++m) {
        const int r = o + n + rows * pr + m;
        *reinterpret_cast<float4 *>(Lp + r * 64 + lsw(r, o + 4 * pc)) =
            make_float4(-acc[m][0], -acc[m][1], -acc[m][2], -acc[m][3]);
    }
    __syncthreads();
}

// ===================================================================== phase 1
constexpr int P1_THREADS = 128;
constexpr uint32_t P1_SMEM = 3 * 32768 + 1024;  // K, V, Q/L/A regions + alignment slack

__global__ void __launch_bounds__(P1_THREADS, 2)
intra_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mv, const TcParams p, long n_pairs) {
    extern __shared__ unsigned char smraw[];
    __shared__ uint64_t bars[3];
    __shared__ uint32_t tslot;
    __shared__ float sG[128], sBeta[128], sCarry[4];
    __shared__ int sAbort;

    unsigned char *sm = align1024(smraw);
    // KQ: two 64-feature slabs of 32 KB, each [K rows 0..127 | Q rows 0..127]
    // (128-byte rows, 128-byte swizzle), so that [K; Q] is one N = 256
    // operand.  After the Gram products the Q half of slab p holds chunk p's
    // fp32 L / T and then slab p of the bf16 operand T diag(beta).
    unsigned char *KQ = sm;
    unsigned char *sV = sm + 65536;   // [2 slabs][128 rows][128 B]

    const int tid0 = threadIdx.x;
    if (status_bad(p.status)) return;

    if (tid0 == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_mbar_init();
        sAbort = 0;
    }
    if ((tid0 >> 5) == 0) {
        tmem_alloc(&tslot, 256);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();

    // Persistent: work items are (pair of chunks, head), head fastest, so that
    // CTAs running side by side read the same token rows of different heads.
    const long n_items = n_pairs * p.H;
    uint32_t ph = 0;   // mbarrier phase parity of this CTA's current item
    for (long item = blockIdx.x; item < n_items; item += gridDim.x) {
    // The thread index is re-read through an opaque move every item so that
    // the compiler does not hoist (and keep live) the many thread-dependent
    // shared-memory addresses across items.
    int tid = tid0;
    asm volatile("" : "+r"(tid));
    const int warp = tid >> 5, lane = tid & 31;
    const int slot = tid >> 6, t = tid & 63;
    const uint32_t tb = tslot;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const long pair = item / p.H;
    const int h = (int)(item % p.H);
    int seq0, seq1, nc0, nc1;
    long r00, r01;
    const bool v0 = slot_info(p, 2 * pair, seq0, r00, nc0);
    const bool v1 = slot_info(p, 2 * pair + 1, seq1, r01, nc1);
    if (!v0) { nc0 = 0; r00 = 0; }
    if (!v1) { nc1 = 0; r01 = 0; }
    if (!v0 && !v1) continue;
    const int nc = slot ? nc1 : nc0;
    const bool vslot = slot ? v1 : v0;

    if (tid == 0) {
        mbar_expect_tx(&bars[0], 3u * 32768u);
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int z = (int)(q ? r01 : r00);
                tma_load_3d(KQ + s * 32768 + q * 8192, &mk, &bars[0], 64 * s, h, z);
                tma_load_3d(KQ + s * 32768 + 16384 + q * 8192, &mq, &bars[0], 64 * s, h, z);
                tma_load_3d(sV + s * 16384 + q * 8192, &mv, &bars[0], 64 * s, h, z);
            }
    }

    // ---- decay: g = inclusive prefix sum of log alpha within each chunk ----
    float a = 1.f, et = 0.f;
    if (t < nc) {
        const size_t row = (size_t)((slot ? r01 : r00) + t) * p.H + h;
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
    if (!mbar_wait(&bars[0], ph)) {
        sAbort = 1;
        set_status(p.status, kDevTimeout);
    }
    __syncthreads();
    const bool abort1 = sAbort != 0;
    if (tid == 0 && !abort1) {
        tc_fence_after();
        // [K K^T | K Q^T]: A = K (128 tokens), B = [K; Q] (256 rows), K = 128 features
        const uint32_t idesc = idesc_bf16_f32(128, 256, false, false);
        const uint32_t aKQ = smem_u32(KQ);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 32768 + (ks & 3) * 32;
            mma_bf16(tb + 0, sdesc_sw128(aKQ + off, 16, 1024), sdesc_sw128(aKQ + off, 16, 1024),
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
                const uint4 v = *reinterpret_cast<const uint4 *>(KQ + s * 32768 +
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

    // ---- epilogue 1: L = strict_lower(beta Gamma o KK^T) (fp32 smem) from row t of
    //      K K^T; row s of (K Q^T) gives row s of A^T, A = lower(Gamma o QK^T) ----
    bool ok = !abort1 && mbar_wait(&bars[1], ph);
    if (!abort1 && !ok) set_status(p.status, kDevTimeout);
    tc_fence_after();
    const float gt = sG[tid];
    const float bt = sBeta[tid];
    const int cb = slot * 64;
    const long gidx0 = 2L * pair + slot;
    const size_t slot_row = (size_t)(gidx0 * p.H + h) * C + t;   // row of this token in the ws
    if (ok) {
        float *Lrow = lslot(KQ, slot) + t * 64;
#pragma unroll 1
        for (int g16 = 0; g16 < 4; ++g16) {
            uint32_t r[16];
            tmem_ld16(tb + lane_base + cb + g16 * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                float v4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = g16 * 16 + i + e;
                    v4[e] = (s < t && t < nc) ? bt * __expf(gt - sG[cb + s]) * __uint_as_float(r[i + e])
                                              : 0.f;
                }
                *reinterpret_cast<float4 *>(Lrow + lsw(t, g16 * 16 + i)) =
                    make_float4(v4[0], v4[1], v4[2], v4[3]);
            }
        }
#pragma unroll 1
        for (int g16 = 0; g16 < 4; ++g16) {
            uint32_t r[16];
            tmem_ld16(tb + lane_base + 128 + cb + g16 * 16, r);
            tmem_ld_wait();
            // this thread's token is the key s = t; the columns are queries u
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const int u = g16 * 16 + i;
                const float a0 = (t <= u && u < nc)
                                     ? __expf(sG[cb + u] - gt) * __uint_as_float(r[i]) : 0.f;
                const float a1 = (t <= u + 1 && u + 1 < nc)
                                     ? __expf(sG[cb + u + 1] - gt) * __uint_as_float(r[i + 1]) : 0.f;
                pk[i / 2] = pack_bf2(a0, a1);
            }
            if (vslot) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.A_ws + slot_row * 64 + g16 * 16);
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
        }
        // K row -> diag(exp g) K; rows past the chunk's end (another
        // sequence's tokens or TMA zero fill) are cleared in K and V so that
        // nothing from them can reach the products.
        // The state pass needs diag(exp(g_C - g)) K; it goes to the workspace.
        const float gam_t = __expf(gt);
        const float gam_c = __expf(sG[cb + C - 1] - gt);
        const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
        uint4 *kt_row = reinterpret_cast<uint4 *>(p.Kt_ws + slot_row * D);
#pragma unroll 1
        for (int s = 0; s < 2; ++s)
#pragma unroll 2
            for (int ch = 0; ch < 8; ++ch) {
                uint4 *pk4 = reinterpret_cast<uint4 *>(KQ + s * 32768 + sw128_offset(tid, ch * 8));
                if (t < nc) {
                    const uint4 v = *pk4;
                    *pk4 = make_uint4(pack_bf2(gam_t * bf_lo(v.x), gam_t * bf_hi(v.x)),
                                      pack_bf2(gam_t * bf_lo(v.y), gam_t * bf_hi(v.y)),
                                      pack_bf2(gam_t * bf_lo(v.z), gam_t * bf_hi(v.z)),
                                      pack_bf2(gam_t * bf_lo(v.w), gam_t * bf_hi(v.w)));
                    if (vslot)
                        kt_row[s * 8 + ch] = make_uint4(pack_bf2(gam_c * bf_lo(v.x), gam_c * bf_hi(v.x)),
                                                        pack_bf2(gam_c * bf_lo(v.y), gam_c * bf_hi(v.y)),
                                                        pack_bf2(gam_c * bf_lo(v.z), gam_c * bf_hi(v.z)),
                                                        pack_bf2(gam_c * bf_lo(v.w), gam_c * bf_hi(v.w)));
                } else {
                    if (vslot) kt_row[s * 8 + ch] = zero4;
                    *pk4 = zero4;
                    *reinterpret_cast<uint4 *>(sV + s * 16384 + sw128_offset(tid, ch * 8)) = zero4;
                }
            }
    }
    if (!ok) sAbort = 1;
    __syncthreads();
    const bool abort2 = sAbort != 0;

    // ---- T = (I + L)^{-1}, built up in block sizes 16 -> 32 -> 64: the
    //      diagonal 16 x 16 blocks by forward substitution, then at each level
    //      [[D1, 0], [X, D2]] with X = -D2 L21 D1 from two small products ----
    {
        // diagonal 16 x 16 blocks: 16 threads per block, one column each
        const int p = tid >> 6, blk = (tid >> 4) & 3, c = tid & 15, o = 16 * blk;
        float *Lb = lslot(KQ, p) + o * 64;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float *Lr = Lb + r * 64;
            float a0 = (r == c) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                if (4 * s4 < r) {
                    const float4 l = *reinterpret_cast<const float4 *>(Lr + lsw(o + r, o + 4 * s4));
                    a0 = fmaf(-l.x, x[4 * s4], a0);
                    if (4 * s4 + 1 < r) a1 = fmaf(-l.y, x[4 * s4 + 1], a1);
                    if (4 * s4 + 2 < r) a0 = fmaf(-l.z, x[4 * s4 + 2], a0);
                    if (4 * s4 + 3 < r) a1 = fmaf(-l.w, x[4 * s4 + 3], a1);
                }
            }
            x[r] = a0 + a1;
        }
        __syncthreads();  // the diagonal blocks of L have been read
#pragma unroll
        for (int r = 0; r < 16; ++r) Lb[r * 64 + lsw(o + r, o + c)] = x[r];
        __syncthreads();
    }
    merge_level<16>(KQ, tid);   // 32 x 32 diagonal blocks
    merge_level<32>(KQ, tid);   // the whole 64 x 64 inverse

    // ---- A operand = T diag(beta) in bf16, block diagonal over the two chunks ----
    {
        const float *Trow = lslot(KQ, slot) + t * 64;
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 v = *reinterpret_cast<const float4 *>(Trow + lsw(t, 4 * i));
            const float *bs = sBeta + slot * 64 + 4 * i;
            pk[2 * i] = pack_bf2(v.x * bs[0], v.y * bs[1]);
            pk[2 * i + 1] = pack_bf2(v.z * bs[2], v.w * bs[3]);
        }
        __syncthreads();  // T fully read; its region becomes the bf16 A tile
        unsigned char *own = KQ + slot * 32768 + 16384, *other = KQ + (1 - slot) * 32768 + 16384;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            *reinterpret_cast<uint4 *>(own + sw128_offset(tid, ch * 8)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            *reinterpret_cast<uint4 *>(other + sw128_offset(tid, ch * 8)) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && !abort2) {
        tc_fence_after();
        const uint32_t aA = smem_u32(KQ + 16384), aK = smem_u32(KQ), aV = smem_u32(sV);
        // W = (T diag beta) (diag(exp g) K): M = 128 tokens, N = 128, K = 128 tokens;
        // A slabs (one per chunk's columns) at 32 KB; B = diag(exp g) K MN-major
        // (rows = tokens), its two 64-feature n-blocks 32 KB apart.
        const uint32_t id_w = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16(tb + 0, sdesc_sw128(aA + (ks >> 2) * 32768 + (ks & 3) * 32, 16, 1024),
                     sdesc_sw128(aK + ks * 2048, 32768, 1024), id_w, ks > 0);
        // U~^T = V^T (T diag beta)^T: M = 128 features (A = V, MN-major), N = 128
        // tokens (B = the same T diag beta tile, K-major), K = 128 tokens.
        const uint32_t id_u = idesc_bf16_f32(128, 128, true, false);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16(tb + 128, sdesc_sw128(aV + ks * 2048, 16384, 1024),
                     sdesc_sw128(aA + (ks >> 2) * 32768 + (ks & 3) * 32, 16, 1024), id_u, ks > 0);
        mma_commit(&bars[2]);
    }
    __syncthreads();

    // ---- epilogue 2: W rows, U~^T rows (bf16) and g to the workspace ----
    ok = !abort2 && mbar_wait(&bars[2], ph);
    if (!abort2 && !ok) set_status(p.status, kDevTimeout);
    tc_fence_after();
    if (ok) {
        if (vslot) {
            __nv_bfloat16 *dst_row = p.W_ws + slot_row * D;
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t r[32];
                tmem_ld32(tb + lane_base + c4 * 32, r);
                tmem_ld_wait();
                store_bf16x32(dst_row + c4 * 32, r);
            }
            p.eg_ws[slot_row] = __expf(gt);
        }
        // lane j of U~^T holds feature j for the tokens of both chunks
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
            uint32_t r0[32], r1[32];
            tmem_ld32(tb + lane_base + 128 + q * 64, r0);
            tmem_ld32(tb + lane_base + 128 + q * 64 + 32, r1);
            tmem_ld_wait();
            if (q ? v1 : v0) {
                __nv_bfloat16 *dst = p.UT_ws + ((size_t)((2L * pair + q) * p.H + h) * D + tid) * C;
                store_bf16x32(dst, r0);
                store_bf16x32(dst + 32, r1);
            }
        }
    }
    tc_fence_before();
    __syncthreads();   // smem and TMEM free for the next item
    ph ^= 1u;
    if (sAbort) break;
    }  // items
    if ((tid0 >> 5) == 0) tmem_dealloc(tslot, 256);
}

// ===================================================================== phase 2
// Warp roles:
//   warps 0-7 ("main"): the serial chain and the outputs; thread (j, half)
//             owns dv index j (its TMEM lane) and tokens [32*half, +32) /
//             state rows [64*half, +64).
//   warp 8    ("issuer"): issues every MMA and TMA load from lane 0; the warp
//             waits on its barriers converged.
// Per chunk the tensor core runs two wide products:
//   [P^T | X^T] = S^T [W ; Q]^T                                M=128, N=128, K=128
//   [Z^T | Y^T] = U^T [diag(exp(g_C - g)) K | A^T]             M=128, N=192, K=64
// with U^T = U~^T - P^T, S^T <- exp(g_C) S^T + Z^T and
// O^T = X^T diag(exp g) + Y^T.  diag(exp(g_C - g)) K and exp(g) come from
// phase 1.  The bf16 A operands S^T and U^T live in tensor memory, which
// leaves shared memory for three chunk stages in flight.
constexpr int P2_MAIN = 256, P2_THREADS = P2_MAIN + 32;
constexpr int NSTAGE = 3;
// Stage layout (one chunk):
//   WQ: two 64-feature slabs of 16 KB, each [W rows 0..63 | Q rows 0..63]
//   KA: K~ slab 0, K~ slab 1, A^T (8 KB each): MN-major n-blocks 8 KB apart
//   U:  U~^T [128][64];  EG: exp(g) [64]
constexpr uint32_t ST_WQ = 0, ST_KA = 32768, ST_A = 49152, ST_U = 57344, ST_EG = 73728,
                   ST_BYTES = 74752;
constexpr uint32_t ST_TX = 16384u * 4u + 8192u + 256u;  // bytes a stage receives
constexpr uint32_t P2_SMEM = NSTAGE * ST_BYTES + 1024;

// TMEM columns (M = 128 lanes = dv): fp32 [P^T | X^T] 0..127; fp32
// [Z^T | Y^T] 128..319; bf16 S^T (128 packed as 64) 320..383; bf16 U^T (64
// packed as 32) 384..415.
constexpr uint32_t TM_PX = 0, TM_ZY = 128, TM_S = 320, TM_U = 384;

__device__ __forceinline__ void issue_stage(unsigned char *st, uint64_t *bar,
                                            const CUtensorMap *mq, const CUtensorMap *mkt,
                                            const CUtensorMap *mw, const CUtensorMap *mu,
                                            const CUtensorMap *ma, const float *eg_src, int h,
                                            int row0, int slot) {
    mbar_expect_tx(bar, ST_TX);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        tma_load_2d(st + ST_WQ + s * 16384, mw, bar, 64 * s, slot * C);
        tma_load_3d(st + ST_WQ + s * 16384 + 8192, mq, bar, 64 * s, h, row0);
        tma_load_2d(st + ST_KA + s * 8192, mkt, bar, 64 * s, slot * C);
    }
    tma_load_2d(st + ST_A, ma, bar, 0, slot * C);
    tma_load_2d(st + ST_U, mu, bar, 0, slot * D);
    bulk_load(st + ST_EG, eg_src, 256, bar);
}

// Main warps: bf16 copy of the 64 state values S[64*half + i][j] into the
// TMEM operand S^T (row j, packed columns 32*half ..).
__device__ __forceinline__ void store_state_bf16(uint32_t taddr, const float (&Sr)[64]) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf2(Sr[32 * hh + 2 * i], Sr[32 * hh + 2 * i + 1]);
        tmem_st16(taddr + 16 * hh, pk);
    }
}

__global__ void __launch_bounds__(P2_THREADS, 1)
state_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mkt,
             const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
             const __grid_constant__ CUtensorMap ma, const TcParams p) {
    extern __shared__ unsigned char smraw[];
    __shared__ uint64_t bar_ld[NSTAGE];
    __shared__ uint64_t bar_p, bar_u, bar_zy, bar_sready;
    __shared__ uint32_t tslot;
    __shared__ int sAbort;

    unsigned char *sm = align1024(smraw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    const int half = (warp >> 2) & 1;           // main warps only
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
        for (int i = 0; i < NSTAGE; ++i) mbar_init(&bar_ld[i], 1);
        mbar_init(&bar_p, 1);
        mbar_init(&bar_u, P2_MAIN);
        mbar_init(&bar_zy, 1);
        mbar_init(&bar_sready, P2_MAIN);
        fence_mbar_init();
        sAbort = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tslot;

    // fp32 master state (main warps): S[i][j] for i in [64*half, 64*half+64)
    float Sr[64];
    if (tid < P2_MAIN) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
            Sr[i] = p.S0 ? p.S0[sbase + (size_t)(64 * half + i) * D + j] : 0.f;
        store_state_bf16(tb + lane_base + TM_S + 32 * half, Sr);
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    auto fail = [&]() {
        sAbort = 1;
        set_status(p.status, kDevTimeout);
    };

    if (warp == 8) {
        // ----------------------------------------------------------------- issuer
        const uint32_t id_px = idesc_bf16_f32(128, 128, false, false);
        const uint32_t id_zy = idesc_bf16_f32(128, 192, false, true);
        if (lane == 0) {
            for (int c = 0; c < NSTAGE && c < nch; ++c) {
                const long slot = (chunk0 + c) * p.H + h;
                issue_stage(sm + c * ST_BYTES, &bar_ld[c], &mq, &mkt, &mw, &mu, &ma,
                            p.eg_ws + slot * C, h, (int)(start + (long)c * C), (int)slot);
            }
        }
        __syncwarp();
        for (int c = 0; c < nch; ++c) {
            const int b = c % NSTAGE;
            unsigned char *st = sm + b * ST_BYTES;
            const uint32_t par = (uint32_t)(c & 1), par_st = (uint32_t)((c / NSTAGE) & 1);
            bool ok = mbar_wait(&bar_ld[b], par_st);
            if (ok && c >= 1) ok = mbar_wait(&bar_sready, par ^ 1u);  // chunk c-1 finished
            if (!__all_sync(0xffffffffu, ok)) { fail(); break; }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t aWQ = smem_u32(st + ST_WQ);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ta(tb + TM_PX, tb + TM_S + 8 * ks,
                                sdesc_sw128(aWQ + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                id_px, ks > 0);
                mma_commit(&bar_p);
            }
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_u, par))) { fail(); break; }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t aKA = smem_u32(st + ST_KA);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ta(tb + TM_ZY, tb + TM_U + 8 * ks,
                                sdesc_sw128(aKA + ks * 2048, 8192, 1024), id_zy, ks > 0);
                mma_commit(&bar_zy);
            }
            __syncwarp();
            // both products have read this stage: refill it with chunk c + NSTAGE
            if (c + NSTAGE < nch) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_zy, par))) { fail(); break; }
                if (lane == 0) {
                    const long slot = (chunk0 + c + NSTAGE) * p.H + h;
                    issue_stage(st, &bar_ld[b], &mq, &mkt, &mw, &mu, &ma, p.eg_ws + slot * C, h,
                                (int)(start + (long)(c + NSTAGE) * C), (int)slot);
                }
                __syncwarp();
            }
        }
    } else {
        // ----------------------------------------------------------------- main
        const size_t rs = (size_t)p.H * D;
        for (int c = 0; c < nch; ++c) {
            const int b = c % NSTAGE;
            unsigned char *st = sm + b * ST_BYTES;
            const uint32_t par = (uint32_t)(c & 1), par_st = (uint32_t)((c / NSTAGE) & 1);
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_ld[b], par_st) && mbar_wait(&bar_p, par))) {
                fail();
                break;
            }
            tc_fence_after();
            const float *eg = reinterpret_cast<const float *>(st + ST_EG);
            const float egC = eg[C - 1];
            // ---- U^T = U~^T - P^T for tokens [32*half, 32*half + 32) -> TMEM (bf16) ----
            {
                uint32_t r[32];
                tmem_ld32(tb + lane_base + TM_PX + half * 32, r);
                tmem_ld_wait();
                const unsigned char *sU = st + ST_U;
                uint32_t pk[16];
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(sU + sw128_offset(j, half * 32 + v4 * 8));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        pk[4 * v4 + e] = pack_bf2(bf_lo(w[e]) - __uint_as_float(r[8 * v4 + 2 * e]),
                                                  bf_hi(w[e]) - __uint_as_float(r[8 * v4 + 2 * e + 1]));
                }
                tmem_st16(tb + lane_base + TM_U + 16 * half, pk);
                tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive(&bar_u);

            if (!__all_sync(0xffffffffu, mbar_wait(&bar_zy, par))) { fail(); break; }
            tc_fence_after();
            // ---- S^T <- exp(g_C) S^T + Z^T ; new bf16 copy of S^T in TMEM ----
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r[32];
                tmem_ld32(tb + lane_base + TM_ZY + half * 64 + c2 * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    Sr[c2 * 32 + i] = fmaf(egC, Sr[c2 * 32 + i], __uint_as_float(r[i]));
            }
            store_state_bf16(tb + lane_base + TM_S + 32 * half, Sr);
            // ---- O = diag(exp g) X + Y for this chunk's tokens, read before the next
            //      product overwrites X^T, stored while that product runs ----
            uint32_t opk[16];
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                uint32_t xr[16], yr[16];
                tmem_ld16(tb + lane_base + TM_PX + 64 + half * 32 + 16 * q2, xr);
                tmem_ld16(tb + lane_base + TM_ZY + 128 + half * 32 + 16 * q2, yr);
                tmem_ld_wait();
                const float *egt = eg + 32 * half + 16 * q2;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    opk[8 * q2 + i] =
                        pack_bf2(fmaf(egt[2 * i], __uint_as_float(xr[2 * i]), __uint_as_float(yr[2 * i])),
                                 fmaf(egt[2 * i + 1], __uint_as_float(xr[2 * i + 1]),
                                      __uint_as_float(yr[2 * i + 1])));
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar_sready);
            const int nc = (int)min((long)C, len - (long)c * C);
            __nv_bfloat16 *dst = p.o + (size_t)(start + (long)c * C + 32 * half) * rs + (size_t)h * D + j;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = 32 * half + 2 * i;
                if (t < nc) dst[(size_t)(2 * i) * rs] = __ushort_as_bfloat16((unsigned short)(opk[i] & 0xffffu));
                if (t + 1 < nc)
                    dst[(size_t)(2 * i + 1) * rs] = __ushort_as_bfloat16((unsigned short)(opk[i] >> 16));
            }
        }
        if (!sAbort && p.S_T) {
#pragma unroll
            for (int i = 0; i < 64; ++i) p.S_T[sbase + (size_t)(64 * half + i) * D + j] = Sr[i];
        }
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

bool map_2d(CUtensorMap *m, const void *base, int cols, long rows, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                       strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (persistent grids).
int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

struct WsLayout {
    size_t meta, g, W, U, A, Kt, total;
};

WsLayout layout(long n_chunks, int H, int n_seq) {
    const size_t slots = (size_t)n_chunks * H;
    WsLayout L;
    L.meta = 0;
    L.g = align_up(((size_t)2 * n_seq + 1) * sizeof(int), 1024);
    L.W = L.g + align_up(slots * C * sizeof(float), 1024);
    L.U = L.W + slots * C * D * 2;
    L.A = L.U + slots * C * D * 2;
    L.Kt = L.A + slots * C * C * 2;
    L.total = L.Kt + slots * C * D * 2;
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
    tp.eg_ws = reinterpret_cast<float *>(ws + L.g);
    tp.Kt_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.Kt);
    tp.W_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.W);
    tp.UT_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.U);
    tp.A_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.A);
    int *chunk_prefix = reinterpret_cast<int *>(ws + L.meta);
    int *order = chunk_prefix + p.n_seq + 1;
    tp.chunk_prefix = p.cu_seqlens ? chunk_prefix : nullptr;
    tp.order = p.cu_seqlens ? order : nullptr;

    CUtensorMap mq, mk, mv, mw, mu, ma, mkt;
    const long slots = n_chunks_upper * p.H;
    if (!map_3d_rows(&mq, p.q, p.H, p.total_T) || !map_3d_rows(&mk, p.k, p.H, p.total_T) ||
        !map_3d_rows(&mv, p.v, p.H, p.total_T) || !map_2d(&mw, tp.W_ws, D, slots * C, C) ||
        !map_2d(&mu, tp.UT_ws, C, slots * D, D) || !map_2d(&ma, tp.A_ws, C, slots * C, C) ||
        !map_2d(&mkt, tp.Kt_ws, D, slots * C, C))
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
    const long n_pairs = (n_chunks_upper + 1) / 2;
    const long n_items = n_pairs * p.H;
    const long grid1 = n_items < 2L * sm_count() ? n_items : 2L * sm_count();
    intra_kernel<<<(unsigned)grid1, P1_THREADS, P1_SMEM, s>>>(mq, mk, mv, tp, n_pairs);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    state_kernel<<<(unsigned)(p.n_seq * p.H), P2_THREADS, P2_SMEM, s>>>(mq, mkt, mw, mu, ma, tp);
    note_launch();
    return cudaGetLastError();
}

}  // namespace kla
