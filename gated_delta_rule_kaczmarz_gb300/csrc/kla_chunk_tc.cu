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
// W = (T diag beta)(diag(exp g) K) and U~ = (T diag beta) V with two MMAs.
// W, U~, A^T (bf16) and g (fp32) go to the caller's workspace.
//
// Phase 2 (state_kernel) walks the chunks of one (sequence, head) in order;
// the two 64-column halves of the state run in two CTAs, since the columns
// of S evolve independently.  Per chunk, with S_b the CTA's dk x 64 slice:
//   [X | P] = [Q ; W] S_b ;  U = U~_b - P
//   S_b <- exp(g_C) S_b + K^T (diag(exp(g_C - g)) U)   (S_b fp32 in TMEM)
//   Y = A U ;  O_b = diag(exp g) X + Y
// The serial chain is [X | P] -> U -> K^T U' -> S_b to shared memory; one
// warp issues the chain's MMAs, another Y, a third the TMA loads (three
// chunks in flight), and the outputs of a chunk are formed and stored while
// the next chunk's first product runs.

// All waits are bounded (kla_tc.cuh); a wait that gives up sets the status
// word to a timeout code and the CTA leaves after releasing TMEM.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>

#include "kla_internal.h"
#include "kla_tc.cuh"
#include "kla_tmap.h"

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
    const int2 *chunk_tab;     // varlen only: (first token row, tokens) of each chunk
    const int *order;          // varlen only: sequences by decreasing length, [N]
    unsigned *status;
    float *g_ws;               // [slots][64]        g_t (in-chunk cumulative log decay)
    __nv_bfloat16 *W_ws;       // [slots][64][128]
    __nv_bfloat16 *U_ws;       // [slots][64][128]   U~
    __nv_bfloat16 *A_ws;       // [slots][64 keys s][64 queries t]  A^T
    int beta_mode;             // 0: beta = eta / (||k||^2 + eps); 1: beta = eta
    // Sequence split (fixed length): every sequence of seg_T tokens (seg_nch
    // chunks) is run as seg_P virtual sequences (segments) of whole 128-token
    // tiles: the first seg_r segments hold seg_q + 1 tiles, the others seg_q.
    // State CTAs [0, phi_first) run the state pass of the virtual sequences
    // (S0 only for the first segment); CTAs from phi_first on run the
    // transition pass of the later segments (S0 = I, U~ read as 0), whose
    // outputs are Q_corr rows (o_phi) and Phi (S_T_phi).
    int seg_P, phi_first;
    int seg_T, seg_nch, seg_q, seg_r;
    __nv_bfloat16 *o_phi;
    float *S_T_phi;
    // Recording for the backward pass: the state at every chunk start (per
    // slot = chunk * H + head, two 16 KB images of the bf16 operand tiles of
    // its column halves, copied from shared memory as the state pass holds
    // them) and T of every chunk slot ([slots][64][64] bf16); o may then be
    // null.
    unsigned char *S_chk;
    __nv_bfloat16 *T_chk;
    unsigned *flags;           // fused launch: one ready flag per work item, then the work-item
                               // counter (all zeroed per call)
    int n_units;               // fused launch: sequences x heads
    // fused launch: the bound (clock64 cycles) of every wait on a ready flag,
    // and an optional word that nothing sets, zeroed per call, on which the
    // state pass waits once before its first load (a test of the timeout
    // path; nullptr in normal calls)
    long long flag_wait_limit;
    const unsigned *test_gate;
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

// Segment s of a split sequence: its first 128-token tile and its tile count.
__host__ __device__ __forceinline__ void seg_tiles(int q, int r, int s, int &tile0, int &ntiles) {
    tile0 = s * q + (s < r ? s : r);
    ntiles = q + (s < r ? 1 : 0);
}

// Chunk slot g: its first token row and valid length.  False when g lies
// beyond the last chunk (the grid is sized by an upper bound).
__device__ __forceinline__ bool slot_info(const TcParams &p, long g, long &row0, int &nc) {
    if (p.chunk_prefix == nullptr) {
        if (p.nch_fixed <= 0) return false;
        // 32-bit division: chunk slots stay below 2^31 (the host checks)
        const uint32_t q = (uint32_t)g / (uint32_t)p.nch_fixed;
        if ((int)q >= p.n_seq) return false;
        const int c = (int)((uint32_t)g - q * (uint32_t)p.nch_fixed);
        row0 = (long)q * p.T + (long)c * C;
        nc = min(C, p.T - c * C);
        return true;
    }
    // the chunk table written by the preparation kernel (one entry past the
    // last chunk slot, so that the read needs no bound first)
    const int total = p.chunk_prefix[p.n_seq];
    const int2 e = p.chunk_tab[g];
    if (g >= total) return false;
    row0 = e.x;
    nc = e.y;
    return nc > 0;
}

// 2^x with the hardware approximation (PTX ex2.approx, relative error about
// 2^-22; 0 for large negative x).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // a -> low half
    return *reinterpret_cast<const uint32_t *>(&v);
}
// A bf16 pair as two floats (low half first).
__device__ __forceinline__ float2 bf2_f2(uint32_t u) { return make_float2(bf_lo(u), bf_hi(u)); }
// Two fp32 lanes per instruction (each lane rounded as the scalar operation).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 bcast2(float a) { return make_float2(a, a); }

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

constexpr int P1_THREADS = 256;

// The first doubling step (n = 16: blocks of 32 at offsets o = 0, 32 of both
// chunks, four blocks), with the triangular zeros skipped and the work
// balanced: warps 0-3 take blocks 0, 1 and warps 4-7 blocks 2, 3 (lane / 16
// the block, lane % 16 the row or row-and-column).  M = L21 D1: warp w forms
// 4-column block cb (w % 4 for w < 4, 3 - w % 4 after) of all 16 rows from
// rows s >= 4 cb of D1 (4 - cb steps).  X = -D2 M: warp w forms row group j
// (the same rule; 4 rows x 4 column blocks) from columns s <= 4 j + 3 of D2
// (j + 1 steps).  Every warp runs five steps.  M goes through `scratch` in
// rows of 20 floats (float4-aligned, and the row-per-lane stores spread over
// the banks).
__device__ __forceinline__ void merge_mid(unsigned char *kq, float *scratch, int tid, int bar) {
    constexpr int MS = 20;
    const int w = tid >> 5, lane = tid & 31;
    const int sel = w < 4 ? (w & 3) : 3 - (w & 3);
    const int blk = (w < 4 ? 0 : 2) + (lane >> 4);
    const int o = 32 * (blk & 1);
    float *Lp = lslot(kq, blk >> 1);
    float *Mb = scratch + blk * 16 * MS;
    {
        const int cb = sel, rho = lane & 15, r = o + 16 + rho;
        float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll 1
        for (int s4 = cb; s4 < 4; ++s4) {
            const float4 a = *reinterpret_cast<const float4 *>(Lp + r * 64 + lsw(r, o + 4 * s4));
            const float am[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s = o + 4 * s4 + e;
                const float4 b = *reinterpret_cast<const float4 *>(Lp + s * 64 + lsw(s, o + 4 * cb));
                a01 = fma2(bcast2(am[e]), make_float2(b.x, b.y), a01);
                a23 = fma2(bcast2(am[e]), make_float2(b.z, b.w), a23);
            }
        }
        *reinterpret_cast<float4 *>(Mb + rho * MS + 4 * cb) = make_float4(a01.x, a01.y, a23.x, a23.y);
    }
    named_sync(bar, P1_THREADS);  // M complete; L21 no longer read
    {
        const int j = sel, rr = lane & 15, rho = 4 * j + (rr >> 2), cb = rr & 3, r = o + 16 + rho;
        float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll 1
        for (int s4 = 0; s4 <= j; ++s4) {
            const float4 a = *reinterpret_cast<const float4 *>(Lp + r * 64 + lsw(r, o + 16 + 4 * s4));
            const float am[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 b = *reinterpret_cast<const float4 *>(Mb + (4 * s4 + e) * MS + 4 * cb);
                a01 = fma2(bcast2(am[e]), make_float2(b.x, b.y), a01);
                a23 = fma2(bcast2(am[e]), make_float2(b.z, b.w), a23);
            }
        }
        *reinterpret_cast<float4 *>(Lp + r * 64 + lsw(r, o + 4 * cb)) =
            make_float4(-a01.x, -a01.y, -a23.x, -a23.y);
    }
    named_sync(bar, P1_THREADS);
}

// The last doubling step (n = 32, one block per chunk, 128 threads per chunk),
// with the zeros of the triangular factors skipped and the work spread evenly
// over the four warps of a chunk.  M = L21 D1: column c of M needs rows s >= c
// of D1 only, so the thread of L21 row `lane` forms the 4-column blocks w and
// 7 - w of its row (8 - w and w + 1 steps of four rows of D1).  X = -D2 M: row
// r needs columns s <= r of D2 only, so warp w forms the row groups w and
// 7 - w (4 rows each; lane / 8 the row, lane % 8 the column block), again
// w + 1 and 8 - w steps.  M goes through `scratch` with its float4 index
// XORed with (row % 8), which keeps the row-per-lane stores and the row reads
// free of bank conflicts.
__device__ __forceinline__ void merge_top(unsigned char *kq, float *scratch, int tid, int bar) {
    const int p = tid >> 7, w = (tid >> 5) & 3, lane = tid & 31;
    float *Lp = lslot(kq, p);
    float *Mp = scratch + p * 1024;
    {
        const int r = 32 + lane;
#pragma unroll 1
        for (int k = 0; k < 2; ++k) {
            const int cb = k ? 7 - w : w;
            float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int s4 = cb; s4 < 8; ++s4) {
                const float4 a = *reinterpret_cast<const float4 *>(Lp + r * 64 + lsw(r, 4 * s4));
                const float am[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = 4 * s4 + e;
                    const float4 b = *reinterpret_cast<const float4 *>(Lp + s * 64 + lsw(s, 4 * cb));
                    a01 = fma2(bcast2(am[e]), make_float2(b.x, b.y), a01);
                    a23 = fma2(bcast2(am[e]), make_float2(b.z, b.w), a23);
                }
            }
            *reinterpret_cast<float4 *>(Mp + lane * 32 + ((cb ^ (lane & 7)) << 2)) =
                make_float4(a01.x, a01.y, a23.x, a23.y);
        }
    }
    named_sync(bar, P1_THREADS);  // M complete; L21 no longer read
    {
        const int pc = lane & 7;
#pragma unroll 1
        for (int k = 0; k < 2; ++k) {
            const int j = k ? 7 - w : w;
            const int rr = 4 * j + (lane >> 3), r = 32 + rr;
            float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int s4 = 0; s4 <= j; ++s4) {
                const float4 a = *reinterpret_cast<const float4 *>(Lp + r * 64 + lsw(r, 32 + 4 * s4));
                const float am[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = 4 * s4 + e;
                    const float4 b = *reinterpret_cast<const float4 *>(Mp + s * 32 + ((pc ^ (s & 7)) << 2));
                    a01 = fma2(bcast2(am[e]), make_float2(b.x, b.y), a01);
                    a23 = fma2(bcast2(am[e]), make_float2(b.z, b.w), a23);
                }
            }
            *reinterpret_cast<float4 *>(Lp + r * 64 + lsw(r, 4 * pc)) =
                make_float4(-a01.x, -a01.y, -a23.x, -a23.y);
        }
    }
    named_sync(bar, P1_THREADS);
}


// ===================================================================== phase 1
// Two threads per token row r of the item (r = tid % 128, the TMEM lane its
// warp reads): thread half hf = tid / 128 takes one of two column halves of
// every per-row task (64-feature slab hf of K and V; the L rows or the A^T
// rows; 32 of the 64 columns of T diag beta; the W rows or the U~ rows).
// Shared memory of one phase-1 worker: K|Q slabs (64 KB), V (32 KB), the
// inverse's scratch (8 KB), then barriers and per-row scalars.
constexpr uint32_t P1_SMALL = 3 * 32768 + 8192;
constexpr uint32_t P1_REGION = 109568;
static_assert(P1_SMALL + 64 + 4 * 512 <= P1_REGION, "phase-1 region");
constexpr uint32_t P1_SMEM = P1_REGION + 1024;   // + alignment slack
// Longest wait of a follower worker for its leader's signal (a timing hint
// only: past it the follower starts anyway).
constexpr long long kStaggerLimitCycles = 40000;

// Phase-1 worker: 256 threads (tid0 = 0..255) with named barrier `bar` over
// them, shared memory `sm` (1024-aligned, P1_REGION bytes), work items
// item0, item0 + step, ...  kFused: items run chunk-pair-major over all
// (sequence, head) units, and each finished item is published through
// p.flags for the state pass running in the same launch.
//
// `stagger` (optional, shared by the two workers of one CTA) offsets them:
// the leader (stagger_role 1) raises it halfway through its first item, and
// the follower (stagger_role 2) starts its first item only then (or after a
// bounded wait).  Two workers that start together wait for their loads
// together and then compete for the same pipes through every step of the
// item; offset by half an item, one computes while the other loads.
template <bool kFused, bool kRecord = true>
__device__ __forceinline__ void intra_run(const CUtensorMap *mq, const CUtensorMap *mk,
                                          const CUtensorMap *mv, const CUtensorMap *mw,
                                          const CUtensorMap *mu, const TcParams &p, long n_pairs,
                                          unsigned char *sm, int tid0, int bar, long item0,
                                          long step, volatile int *stagger = nullptr,
                                          int stagger_role = 0) {
    // KQ: two 64-feature slabs of 32 KB, each [K rows 0..127 | Q rows 0..127]
    // (128-byte rows, 128-byte swizzle), so that [K; Q] is one N = 256
    // operand.  After the Gram products the Q half of slab p holds chunk p's
    // fp32 L / T and then slab p of the bf16 operand T diag(beta).
    unsigned char *KQ = sm;
    unsigned char *sV = sm + 65536;   // [2 slabs][128 rows][128 B]
    float *scratch = reinterpret_cast<float *>(sm + 98304);   // 8 KB, the inverse's products
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + P1_SMALL);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P1_SMALL + 32);
    volatile int *sAbort = reinterpret_cast<volatile int *>(sm + P1_SMALL + 36);
    volatile long *sItem = reinterpret_cast<volatile long *>(sm + P1_SMALL + 40);
    float *sCarry = reinterpret_cast<float *>(sm + P1_SMALL + 48);
    float *sG = reinterpret_cast<float *>(sm + P1_SMALL + 64);   // g of each token row
    float *sG2 = sG + 128;                                         // g * log2(e)
    float *sBeta = sG2 + 128;
    float *sN2 = sBeta + 128;

    if (tid0 == 0) {
        mbar_init(&bars[0], 1);   // K and Q landed
        mbar_init(&bars[1], 1);   // Gram products done
        mbar_init(&bars[2], 1);   // W and U~ products done
        mbar_init(&bars[3], 1);   // V landed
        fence_mbar_init();
        // an error already reported: read once, so that all the worker's
        // threads agree (threads reading the word at different times might not)
        *sAbort = status_bad(p.status) ? 1 : 0;
    }
    if ((tid0 >> 5) == 0) {
        tmem_alloc(tslot, 256);
        // the allocation permit is per CTA: in the fused launch the CTA's
        // other worker still has to allocate, so it is kept
        if (!kFused) tmem_relinquish();
    }
    named_sync(bar, P1_THREADS);
    tc_fence_after();
    if (*sAbort) {
        if ((tid0 >> 5) == 0) tmem_dealloc(*tslot, 256);
        return;
    }

    // Persistent: work items are (pair of chunks, head), head fastest, so that
    // CTAs running side by side read the same token rows of different heads.
    const long n_items = n_pairs * p.H;
    uint32_t ph = 0;      // mbarrier phase parity of this worker's current item
    long pending = -1;    // fused: item written but not yet published (thread 0)
    bool first = true;    // this worker's first item
    if (stagger && stagger_role == 2) {
        if (tid0 == 0) {
            const long long t0 = clock64();
            while (*stagger == 0 && clock64() - t0 < kStaggerLimitCycles) __nanosleep(64);
        }
        named_sync(bar, P1_THREADS);
    }
    // Work items: item0, item0 + step, ...; or, with step == 0, items item0 +
    // (a global counter's next value), handed out in order as workers free up
    // (the fused launch: a late item then delays only its own unit).
    for (long item = item0;; item += step) {
    if (step == 0) {
        if (tid0 == 0) *sItem = item0 + (long)atomicAdd(p.flags + n_items, 1u);
        named_sync(bar, P1_THREADS);
        item = *sItem;
        named_sync(bar, P1_THREADS);
    }
    if (item >= n_items) break;
    // The thread index is re-read through an opaque move every item so that
    // the compiler does not hoist (and keep live) the many thread-dependent
    // shared-memory addresses across items.
    int tid = tid0;
    asm volatile("" : "+r"(tid));
    const int warp = tid >> 5, lane = tid & 31;
    const int r = tid & 127, hf = tid >> 7;      // token row of the item, column half
    const int slot = r >> 6, t = r & 63;
    const uint32_t tb = *tslot;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    long pair;
    int h;
    // (32-bit divisions: work items stay below 2^31, which the host checks)
    if (kFused) {   // item = (pair within the sequence) * units + (sequence * H + head)
        const uint32_t i32 = (uint32_t)item, pu = i32 / (uint32_t)p.n_units;
        const uint32_t u = i32 - pu * (uint32_t)p.n_units, su = u / (uint32_t)p.H;
        pair = (long)pu + (long)su * (p.nch_fixed / 2);
        h = (int)(u - su * (uint32_t)p.H);
    } else {
        const uint32_t i32 = (uint32_t)item, pq = i32 / (uint32_t)p.H;
        pair = (long)pq;
        h = (int)(i32 - pq * (uint32_t)p.H);
    }
    int nc0, nc1;
    long r00, r01;
    const bool v0 = slot_info(p, 2 * pair, r00, nc0);
    const bool v1 = slot_info(p, 2 * pair + 1, r01, nc1);
    if (!v0) { nc0 = 0; r00 = 0; }
    if (!v1) { nc1 = 0; r01 = 0; }
    if (!v0 && !v1) continue;
    const int nc = slot ? nc1 : nc0;
    const bool vslot = slot ? v1 : v0;

    if (tid == 0) {
        // K and Q first (the Gram products need them); V, needed only by the
        // U~ product, on its own barrier behind them.  The previous item's
        // W / U~ stores read the K halves and V's region: Q is loaded before
        // waiting for them to leave shared memory.
        mbar_expect_tx(&bars[0], 2u * 32768u);
#pragma unroll 1
        for (int q = 0; q < 2; ++q)
#pragma unroll 1
            for (int s = 0; s < 2; ++s)
                tma_load_3d(KQ + s * 32768 + 16384 + q * 8192, mq, &bars[0], 64 * s, h,
                            (int)(q ? r01 : r00));
        bulk_wait_group_read0();
#pragma unroll 1
        for (int q = 0; q < 2; ++q)
#pragma unroll 1
            for (int s = 0; s < 2; ++s)
                tma_load_3d(KQ + s * 32768 + q * 8192, mk, &bars[0], 64 * s, h, (int)(q ? r01 : r00));
        mbar_expect_tx(&bars[3], 32768u);
#pragma unroll 1
        for (int q = 0; q < 2; ++q)
#pragma unroll 1
            for (int s = 0; s < 2; ++s)
                tma_load_3d(sV + s * 16384 + q * 8192, mv, &bars[3], 64 * s, h,
                            (int)(q ? r01 : r00));
        if (kFused && pending >= 0) {   // the previous item's outputs are complete
            bulk_wait_group0();
            fence_proxy_async_global();
            __threadfence();
            st_release_u32(p.flags + pending, 1u);
            pending = -1;
        }
    }

    // ---- decay: g = inclusive prefix sum of log alpha within each chunk
    //      (first thread half; the second half has no per-row gate work) ----
    float et = 0.f;
    double gs = 0.0;
    if (hf == 0) {
        float a = 1.f;
        if (t < nc) {
            const size_t row = (size_t)((slot ? r01 : r00) + t) * p.H + h;
            a = p.alpha ? p.alpha[row] : 1.f;   // no alpha: no decay
            et = p.eta[row];
        }
        gs = (double)logf(a);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double u = __shfl_up_sync(0xffffffffu, gs, off);
            if (lane >= off) gs += u;
        }
        if (lane == 31) sCarry[warp] = (float)gs;
    }
    named_sync(bar, P1_THREADS);
    if (hf == 0) {
        if (warp & 1) gs += (double)sCarry[warp - 1];
        sG[r] = (float)gs;
        sG2[r] = (float)(gs * 1.4426950408889634);
    }

    // ---- tiles landed: Gram products on the tensor cores ----
    if (!mbar_wait(&bars[0], ph)) {
        *sAbort = 1;
        set_status(p.status, kDevTimeout);
    }
    named_sync(bar, P1_THREADS);
    const bool abort1 = *sAbort != 0;
    if (tid == 0 && !abort1) {
        tc_fence_after();
        // [K K^T | K Q^T]: A = K (128 tokens), B = [K; Q] (256 rows), K = 128 features
        const uint32_t idesc = idesc_bf16_f32(128, 256, false, false);
        const uint32_t aKQ = smem_u32(KQ);
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 32768 + (ks & 3) * 32;
            mma_bf16(tb + 0, sdesc_sw128(aKQ + off, 16, 1024), sdesc_sw128(aKQ + off, 16, 1024),
                     idesc, ks > 0);
        }
        mma_commit(&bars[1]);
    }

    // ---- beta_t from the key's squared norm (fp32 over the bf16 values);
    //      each thread half sums one 64-feature slab ----
    float2 n2p = make_float2(0.f, 0.f);   // even and odd features
#pragma unroll 2
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 v = *reinterpret_cast<const uint4 *>(KQ + hf * 32768 + sw128_offset(r, ch * 8));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = bf2_f2(w[i]);
            n2p = fma2(x, x, n2p);
        }
    }
    const float n2 = n2p.x + n2p.y;
    if (hf) sN2[r] = n2;
    named_sync(bar, P1_THREADS);
    float bt = 0.f;
    if (hf == 0) {
        const float den = (n2 + sN2[r]) + p.eps;
        const float b = p.beta_mode ? et : (den != 0.f ? et / den : 0.f);
        bt = t < nc ? b : 0.f;
        sBeta[r] = bt;
    }

    // ---- epilogue 1: L = strict_lower(beta Gamma o KK^T) (fp32 smem) from row t of
    //      K K^T (first half); row s of (K Q^T) gives row s of A^T, A = lower(Gamma o
    //      QK^T) (second half) ----
    bool ok = !abort1 && mbar_wait(&bars[1], ph);
    if (!abort1 && !ok) set_status(p.status, kDevTimeout);
    tc_fence_after();
    const float gt = sG[r];
    const int cb = slot * 64;
    const long gidx0 = 2L * pair + slot;
    const size_t slot_row = (size_t)(gidx0 * p.H + h) * C + t;   // row of this token in the ws
    // Gamma_ts = exp(g_t - g_s) = exp2(g2_t - g2_s) is evaluated for every
    // element (exponent clamped at 0, where the mask discards it) and masked
    // by a select, so that the loop has no data-dependent branch.
    const float gt2 = sG2[r];
    // A warp's 32 rows are all in one half of their chunk (t < 32 or t >= 32,
    // the same for the whole warp), so the column blocks that the triangle
    // leaves empty (L: columns 32..63 of rows t < 32; A^T: columns 0..31 of
    // rows t >= 32) are written as zeros without being formed.
    if (ok) {
        if (hf == 0) {
            float *Lrow = lslot(KQ, slot) + t * 64;
            const int lim = (t < nc) ? t : 0;     // L row t has columns s < t
#pragma unroll 1
            for (int g16 = 0; g16 < 4; ++g16) {
                if (g16 >= 2 && t < 32) {
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4 *>(Lrow + lsw(t, g16 * 16 + i)) =
                            make_float4(0.f, 0.f, 0.f, 0.f);
                    continue;
                }
                uint32_t rr[16];
                tmem_ld16(tb + lane_base + cb + g16 * 16, rr);
                float gs[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 v = *reinterpret_cast<const float4 *>(sG2 + cb + g16 * 16 + 4 * i);
                    gs[4 * i] = v.x; gs[4 * i + 1] = v.y; gs[4 * i + 2] = v.z; gs[4 * i + 3] = v.w;
                }
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    float v4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s = g16 * 16 + i + e;
                        const float ex = ex2_approx(fminf(gt2 - gs[i + e], 0.f));
                        const float x = bt * ex * __uint_as_float(rr[i + e]);
                        v4[e] = (s < lim) ? x : 0.f;
                    }
                    *reinterpret_cast<float4 *>(Lrow + lsw(t, g16 * 16 + i)) =
                        make_float4(v4[0], v4[1], v4[2], v4[3]);
                }
            }
        } else {
            const int hi = nc;                      // A^T row t has columns u in [t, nc)
#pragma unroll 1
            for (int g16 = 0; g16 < 4; ++g16) {
                if (g16 < 2 && t >= 32) {
                    if (vslot) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.A_ws + slot_row * 64 + g16 * 16);
                        dst[0] = make_uint4(0u, 0u, 0u, 0u);
                        dst[1] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    continue;
                }
                uint32_t rr[16];
                tmem_ld16(tb + lane_base + 128 + cb + g16 * 16, rr);
                float gu[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 v = *reinterpret_cast<const float4 *>(sG2 + cb + g16 * 16 + 4 * i);
                    gu[4 * i] = v.x; gu[4 * i + 1] = v.y; gu[4 * i + 2] = v.z; gu[4 * i + 3] = v.w;
                }
                tmem_ld_wait();
                // this thread's token is the key s = t; the columns are queries u
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const int u = g16 * 16 + i;
                    const float x0 = ex2_approx(fminf(gu[i] - gt2, 0.f)) * __uint_as_float(rr[i]);
                    const float x1 = ex2_approx(fminf(gu[i + 1] - gt2, 0.f)) * __uint_as_float(rr[i + 1]);
                    const float a0 = (t <= u && u < hi) ? x0 : 0.f;
                    const float a1 = (t <= u + 1 && u + 1 < hi) ? x1 : 0.f;
                    pk[i / 2] = pack_bf2(a0, a1);
                }
                if (vslot) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.A_ws + slot_row * 64 + g16 * 16);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
        }
        // K row (slab hf) -> diag(exp g) K, in place for the W product; rows
        // past the chunk's end (another sequence's tokens or TMA zero fill)
        // are cleared in K and V so that nothing from them can reach the
        // products.
        const bool live = t < nc;
        const float gam_t = live ? ex2_approx(gt2) : 0.f;
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch) {
            uint4 *pk4 = reinterpret_cast<uint4 *>(KQ + hf * 32768 + sw128_offset(r, ch * 8));
            const uint4 v = *pk4;
            const float2 gg = bcast2(gam_t);
            float2 a0 = mul2(gg, bf2_f2(v.x)), a1 = mul2(gg, bf2_f2(v.y));
            float2 a2 = mul2(gg, bf2_f2(v.z)), a3 = mul2(gg, bf2_f2(v.w));
            uint4 w = make_uint4(pack_bf2(a0.x, a0.y), pack_bf2(a1.x, a1.y),
                                 pack_bf2(a2.x, a2.y), pack_bf2(a3.x, a3.y));
            if (!live) w = make_uint4(0u, 0u, 0u, 0u);
            *pk4 = w;
        }
    }
    if (!ok) *sAbort = 1;
    named_sync(bar, P1_THREADS);
    const bool abort2 = *sAbort != 0;
    if (first && stagger && stagger_role == 1 && tid == 0) *stagger = 1;
    first = false;

    // ---- T = (I + L)^{-1}, built up in block sizes 16 -> 32 -> 64: the
    //      diagonal 16 x 16 blocks by forward substitution (first half of the
    //      threads), then at each level [[D1, 0], [X, D2]] with X = -D2 L21 D1
    //      from two small products (all threads) ----
    {
        // diagonal 16 x 16 blocks: 16 threads per block, one column each
        const int pp = (tid >> 6) & 1, blk = (tid >> 4) & 3, c = tid & 15, o = 16 * blk;
        float *Lb = lslot(KQ, pp) + o * 64;
        float x[16];
        if (hf == 0) {
#pragma unroll
            for (int rw = 0; rw < 16; ++rw) {
                const float *Lr = Lb + rw * 64;
                float a0 = (rw == c) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    if (4 * s4 < rw) {
                        const float4 l = *reinterpret_cast<const float4 *>(Lr + lsw(o + rw, o + 4 * s4));
                        a0 = fmaf(-l.x, x[4 * s4], a0);
                        if (4 * s4 + 1 < rw) a1 = fmaf(-l.y, x[4 * s4 + 1], a1);
                        if (4 * s4 + 2 < rw) a0 = fmaf(-l.z, x[4 * s4 + 2], a0);
                        if (4 * s4 + 3 < rw) a1 = fmaf(-l.w, x[4 * s4 + 3], a1);
                    }
                }
                x[rw] = a0 + a1;
            }
        }
        named_sync(bar, P1_THREADS);  // the diagonal blocks of L have been read
        if (hf == 0) {
#pragma unroll
            for (int rw = 0; rw < 16; ++rw) Lb[rw * 64 + lsw(o + rw, o + c)] = x[rw];
        }
        named_sync(bar, P1_THREADS);
    }
    merge_mid(KQ, scratch, tid, bar);         // 32 x 32 diagonal blocks
    merge_top(KQ, scratch, tid, bar);         // the whole 64 x 64 inverse

    // ---- V landed; rows past the chunk's end (another sequence's tokens or
    //      TMA zero fill) are cleared so that nothing from them reaches U~ ----
    if (!abort2 && !mbar_wait(&bars[3], ph)) {
        *sAbort = 1;
        set_status(p.status, kDevTimeout);
    }
    if (t >= nc) {
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4 *>(sV + hf * 16384 + sw128_offset(r, ch * 8)) =
                make_uint4(0u, 0u, 0u, 0u);
    }

    // ---- A operand = T diag(beta) in bf16, block diagonal over the two chunks;
    //      thread half hf converts columns [32 hf, 32 hf + 32) of row t ----
    {
        const float *Trow = lslot(KQ, slot) + t * 64;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c4 = 8 * hf + i;
            const float4 v = *reinterpret_cast<const float4 *>(Trow + lsw(t, 4 * c4));
            const float *bs = sBeta + slot * 64 + 4 * c4;
            pk[2 * i] = pack_bf2(v.x * bs[0], v.y * bs[1]);
            pk[2 * i + 1] = pack_bf2(v.z * bs[2], v.w * bs[3]);
        }
        if (kRecord && p.T_chk && vslot) {   // T row t, columns [32 hf, 32 hf + 32), for the backward
            uint4 *dst = reinterpret_cast<uint4 *>(p.T_chk + slot_row * 64 + 32 * hf);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float4 a = *reinterpret_cast<const float4 *>(Trow + lsw(t, 32 * hf + 8 * q4 + 4 * e));
                    w[2 * e] = pack_bf2(a.x, a.y);
                    w[2 * e + 1] = pack_bf2(a.z, a.w);
                }
                dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        named_sync(bar, P1_THREADS);  // T fully read; its region becomes the bf16 A tile
        unsigned char *own = KQ + slot * 32768 + 16384, *other = KQ + (1 - slot) * 32768 + 16384;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            const int cc = 4 * hf + ch;
            *reinterpret_cast<uint4 *>(own + sw128_offset(r, cc * 8)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            *reinterpret_cast<uint4 *>(other + sw128_offset(r, cc * 8)) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    fence_async_smem();
    tc_fence_before();
    named_sync(bar, P1_THREADS);
    const bool abort3 = *sAbort != 0;   // includes a wait for V that ran out
    if (tid == 0 && !abort3) {
        tc_fence_after();
        const uint32_t aA = smem_u32(KQ + 16384), aK = smem_u32(KQ), aV = smem_u32(sV);
        // W = (T diag beta) (diag(exp g) K): M = 128 tokens, N = 128, K = 128 tokens;
        // A slabs (one per chunk's columns) at 32 KB; B = diag(exp g) K MN-major
        // (rows = tokens), its two 64-feature n-blocks 32 KB apart.
        const uint32_t id_w = idesc_bf16_f32(128, 128, false, true);
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16(tb + 0, sdesc_sw128(aA + (ks >> 2) * 32768 + (ks & 3) * 32, 16, 1024),
                     sdesc_sw128(aK + ks * 2048, 32768, 1024), id_w, ks > 0);
        // U~ = (T diag beta) V: the same A; B = V MN-major, n-blocks 16 KB apart.
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16(tb + 128, sdesc_sw128(aA + (ks >> 2) * 32768 + (ks & 3) * 32, 16, 1024),
                     sdesc_sw128(aV + ks * 2048, 16384, 1024), id_w, ks > 0);
        mma_commit(&bars[2]);
    }
    named_sync(bar, P1_THREADS);

    // ---- epilogue 2: W (first half) and U~ (second half) rows of token row r,
    //      bf16, staged in the now free K and V regions with the 128-byte
    //      swizzle of the tensor maps, then written by TMA stores; g ----
    ok = !abort3 && mbar_wait(&bars[2], ph);
    if (!abort3 && !ok) set_status(p.status, kDevTimeout);
    tc_fence_after();
    if (ok) {
        unsigned char *stg = hf ? sV : KQ;
        const uint32_t slab_stride = hf ? 16384u : 32768u;
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t rr[32];
            tmem_ld32(tb + lane_base + 128 * hf + c4 * 32, rr);
            tmem_ld_wait();
            unsigned char *tile = stg + (c4 >> 1) * slab_stride;
            const int col0 = (32 * c4) & 63;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4 *>(tile + sw128_offset(r, col0 + 8 * k)) = make_uint4(
                    pack_bf2(__uint_as_float(rr[8 * k + 0]), __uint_as_float(rr[8 * k + 1])),
                    pack_bf2(__uint_as_float(rr[8 * k + 2]), __uint_as_float(rr[8 * k + 3])),
                    pack_bf2(__uint_as_float(rr[8 * k + 4]), __uint_as_float(rr[8 * k + 5])),
                    pack_bf2(__uint_as_float(rr[8 * k + 6]), __uint_as_float(rr[8 * k + 7])));
        }
        if (hf == 0 && vslot) p.g_ws[slot_row] = gt;
    }
    if (kFused) __threadfence();   // A^T and g rows before the item is published
    fence_async_smem();
    named_sync(bar, P1_THREADS);
    if (tid == 0 && ok) {
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
            if (!(q ? v1 : v0)) continue;
            const int y = (int)(((2L * pair + q) * p.H + h) * C);
#pragma unroll 1
            for (int s = 0; s < 2; ++s) {
                tma_store_2d(mw, KQ + s * 32768 + q * 8192, 64 * s, y);
                tma_store_2d(mu, sV + s * 16384 + q * 8192, 64 * s, y);
            }
        }
        bulk_commit_group();
        if (kFused) pending = item;
    }
    tc_fence_before();
    named_sync(bar, P1_THREADS);   // smem and TMEM free for the next item
    ph ^= 1u;
    if (*sAbort) break;
    }  // items
    if (stagger && stagger_role == 1 && tid0 == 0) *stagger = 1;   // a leader with no item
    if (tid0 == 0) {
        bulk_wait_group0();   // every TMA store complete before the worker leaves
        if (kFused && pending >= 0) {
            fence_proxy_async_global();
            __threadfence();
            st_release_u32(p.flags + pending, 1u);
        }
    }
    if ((tid0 >> 5) == 0) tmem_dealloc(*tslot, 256);
}

__global__ void __launch_bounds__(P1_THREADS, 2)
intra_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mw,
             const __grid_constant__ CUtensorMap mu, const TcParams p, long n_pairs) {
    extern __shared__ unsigned char smraw[];
    intra_run<false>(&mq, &mk, &mv, &mw, &mu, p, n_pairs, align1024(smraw), (int)threadIdx.x, 1,
                     (long)blockIdx.x, (long)gridDim.x);
}

// ===================================================================== phase 2
// One CTA per (sequence, head, half of dv): the columns of S evolve
// independently (S_t = S~ + beta_t k_t e_t^T with e_t = v_t - S~^T k_t acts
// column by column), so the two 64-column halves of a head's state run on two
// SMs side by side.  Per chunk, with S_b = S[:, j0 : j0 + 64] (dk x 64):
//   [X | P] = [Q ; W] S_b                           M=128, N=64, K=128 (dk)
//   U = U~_b - P,  U' = diag(exp(g_C - g)) U  (bf16 -> shared memory)
//   S_b += K^T U',  Y = A U                          M=128, N=64, K=64 (tokens)
//   O_b = diag(exp g) X + Y
// where A = lower(Gamma o Q K^T), and W, U~, A^T and g come from phase 1; Q
// and K are read from the inputs.  S_b is kept in fp32 in TMEM as the
// accumulator of K^T U': the main warps scale it by exp(g_C) while [X | P]
// runs and copy it to shared memory in bf16 after the product.  The serial
// chain per chunk is one 8-step MMA, the U update, one 4-step MMA and the
// bf16 copy of S_b.
//
// Warp roles: warps 0-7 ("main") own TMEM lane L = 32 (warp % 4) + lane
// (= dk row L of S_b, = token L of X / Y for L < 64, = token L - 64 of P for
// L >= 64) and the 32 columns [32 hf, 32 hf + 32) of the tile, hf = warp / 4;
// warp 8 issues the chain's MMAs from lane 0; warp 9 issues the stage loads
// (and, in the fused launch, waits for the ready flags); warp 10 issues Y.
// An MMA issue waits for room in the tensor pipe (about 50 ns per M = 128
// product whatever N), so the product off the chain has a thread of its own:
// the chain's issuer is then free when the next S_b is published.  The three
// wait converged.
constexpr int P2_MAIN = 256, P2_THREADS = P2_MAIN + 96;
constexpr int NSTAGE = 3;
// Stage layout (one chunk):
//   QW: two 64-feature slabs of 16 KB, each [Q rows 0..63 | W rows 0..63]
//   KT: K slab 0, K slab 1 (8 KB each)
//   A:  A^T [64 keys][64 queries];  U: U~[:, j0 : j0 + 64] [64 tokens][64]
// and, in a separate small region, g [64] per stage.
constexpr uint32_t ST_QW = 0, ST_KT = 32768, ST_A = 49152, ST_U = 57344, ST_BYTES = 65536;
constexpr uint32_t ST_TX = 32768u + 16384u + 8192u + 8192u + 256u;  // bytes a stage receives
// After the stages: the bf16 MMA operands S_b [128 dk rows][64], U and U'
// [64 tokens][64] (MN-major, 128-byte swizzle), then g of each stage.
constexpr uint32_t SM_S = NSTAGE * ST_BYTES, SM_U = SM_S + 16384, SM_UZ = SM_U + 8192,
                   SM_G = SM_UZ + 8192;
constexpr uint32_t P2_SMEM = SM_G + NSTAGE * 256 + 1024;

// TMEM columns (fp32, 128 lanes): [X | P] in two buffers, S_b (the
// accumulator of K^T U'), and Y in two buffers (chunk c uses buffer c % 2).
constexpr uint32_t TM_PX = 0, TM_S = 128, TM_Y = 192;

// The same pass with kW dv columns per CTA: kW = 64 (above: two CTAs per
// head, the shorter chain) or kW = 128 (one CTA per head: every product has
// N = 128 for the same MMA count, the element-wise steps take twice as long,
// and half as many CTAs carry the whole state; used where more CTAs than SMs
// would run).  The wide pass has two stages (the stage holds all 128 columns
// of U~) and one Y buffer (TMEM: [X | P] 2 x 128, S_b 128, Y 128 columns).
template <int kW>
struct P2Cfg {
    static constexpr int NST = kW == 64 ? 3 : 2;
    static constexpr int NJ = kW / 64;                 // 64-column slabs of the tile
    // main warps: four per 32-column group (one per TMEM lane quadrant), so
    // that every main thread holds 32 columns of one row whatever kW; then
    // the MMA issuer of the chain, the load warp and the issuer of Y
    static constexpr int NMAIN = kW / 32 * 4;
    static constexpr int THREADS = (NMAIN + 3) * 32;
    static constexpr uint32_t U_BYTES = 64u * kW * 2u;   // U~ of a stage (64-column slabs)
    static constexpr uint32_t ST_BYTES = ST_U + U_BYTES;
    static constexpr uint32_t ST_TX = 32768u + 16384u + 8192u + U_BYTES + 256u;
    static constexpr uint32_t S_SLAB = 128u * 64u * 2u;  // one 64-column slab of S_b
    static constexpr uint32_t U_SLAB = 64u * 64u * 2u;   // one 64-column slab of U, U'
    static constexpr uint32_t SM_S = NST * ST_BYTES, SM_U = SM_S + NJ * S_SLAB,
                              SM_UZ = SM_U + NJ * U_SLAB, SM_G = SM_UZ + NJ * U_SLAB;
    static constexpr uint32_t SMEM = SM_G + NST * 256 + 1024;
    static constexpr uint32_t TM_PX = 0, TM_S = 2 * kW, TM_Y = 3 * kW;
    static constexpr uint32_t Y_STRIDE = kW == 64 ? 64 : 0;   // column offset of Y buffer 1
};
static_assert(P2Cfg<64>::NST == NSTAGE && P2Cfg<64>::ST_BYTES == ST_BYTES &&
                  P2Cfg<64>::ST_TX == ST_TX && P2Cfg<64>::SM_S == SM_S &&
                  P2Cfg<64>::SM_U == SM_U && P2Cfg<64>::SM_UZ == SM_UZ &&
                  P2Cfg<64>::SM_G == SM_G && P2Cfg<64>::SMEM == P2_SMEM &&
                  P2Cfg<64>::TM_PX == TM_PX && P2Cfg<64>::TM_S == TM_S &&
                  P2Cfg<64>::TM_Y == TM_Y,
              "narrow state pass layout");
static_assert(P2Cfg<128>::SMEM <= 232448 && P2Cfg<128>::TM_Y + 128 <= 512, "wide state pass");
static_assert(SM_UZ + 8192 - SM_S == 32768, "S0 staging: the S, U and U' operands of the narrow pass");
static_assert(P2Cfg<64>::THREADS == P2_THREADS, "narrow state pass threads");

template <int kW>
__device__ __forceinline__ void issue_stage(unsigned char *st, float *g_dst, uint64_t *bar,
                                            const CUtensorMap *mq, const CUtensorMap *mk,
                                            const CUtensorMap *mw, const CUtensorMap *mu,
                                            const CUtensorMap *ma, const float *g_src, int h,
                                            int row0, int slot, int j0) {
    mbar_expect_tx(bar, P2Cfg<kW>::ST_TX);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        tma_load_3d(st + ST_QW + s * 16384, mq, bar, 64 * s, h, row0);
        tma_load_2d(st + ST_QW + s * 16384 + 8192, mw, bar, 64 * s, slot * C);
        tma_load_3d(st + ST_KT + s * 8192, mk, bar, 64 * s, h, row0);
    }
    tma_load_2d(st + ST_A, ma, bar, 0, slot * C);
#pragma unroll
    for (int s = 0; s < kW / 64; ++s)
        tma_load_2d(st + ST_U + s * P2Cfg<kW>::U_SLAB, mu, bar, j0 + 64 * s, slot * C);
    bulk_load(g_dst, g_src, 256, bar);
}

// 32 fp32 values -> 32 bf16 at columns [c0, c0 + 32) of row `row` of a
// 128-byte-swizzled tile.
__device__ __forceinline__ void st_row_bf16x32(unsigned char *tile, int row, int c0,
                                               const float (&x)[32]) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, c0 + 8 * k)) =
            make_uint4(pack_bf2(x[8 * k + 0], x[8 * k + 1]), pack_bf2(x[8 * k + 2], x[8 * k + 3]),
                       pack_bf2(x[8 * k + 4], x[8 * k + 5]), pack_bf2(x[8 * k + 6], x[8 * k + 7]));
}

// State pass of CTA `bid` (kW = 64: unit bid / 2, column half bid % 2; kW =
// 128: unit bid) with threads tid = 0 .. P2_THREADS-1 and shared memory `sm`
// (1024-aligned, P2Cfg<kW>::SMEM - 1024 bytes).  kFused: phase 1 runs in the
// same launch, and the load of chunk c waits for the ready flag of the work
// item that holds it.
template <bool kFused, bool kSplit, int kW = 64, bool kRecord = true>
__device__ __forceinline__ void state_run(const CUtensorMap *mq, const CUtensorMap *mk,
                                          const CUtensorMap *mw, const CUtensorMap *mu,
                                          const CUtensorMap *ma, const TcParams &p,
                                          unsigned char *sm, int bid, int tid) {
    using Cf = P2Cfg<kW>;
    constexpr int NS = Cf::NST, NJ = 1;   // one 32-column group per main thread
    constexpr int NMAIN = Cf::NMAIN, NCG = kW / 32;
    __shared__ uint64_t bar_ld[NS];
    __shared__ uint64_t bar_empty[NS];   // the products of a stage's chunk are done
    __shared__ uint64_t bar_px, bar_u, bar_u2, bar_z, bar_s, bar_fin, bar_fin_y;
    __shared__ uint64_t bar_y[2];   // Y of chunk c completes on bar_y[c % 2]
    __shared__ uint32_t tslot;
    __shared__ int sAbort;

    unsigned char *sS = sm + Cf::SM_S, *sU = sm + Cf::SM_U, *sUz = sm + Cf::SM_UZ;
    float *sG = reinterpret_cast<float *>(sm + Cf::SM_G);

    const int warp = tid >> 5, lane = tid & 31;
    const int L = (warp & 3) * 32 + lane;       // TMEM lane (main warps)
    const int hf = (warp >> 2) & (NCG - 1);     // 32-column group (main warps)
    const int c0 = 32 * hf;                     // first of the thread's 32 columns of the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    // transition-pass CTAs: 64 / kW... per (batch, segment >= 1, head), in
    // that order (two 64-column CTAs, or one 128-column CTA, per chain)
    constexpr int CPC = kW == 64 ? 2 : 1;
    const bool phi = kSplit && p.phi_first > 0 && bid >= p.phi_first;
    const int segP = kSplit ? p.seg_P : 1;
    size_t phi_base = 0;
    if (phi) {
        const int k = bid - p.phi_first, idx = k / CPC;
        const int hh = idx % p.H, r = idx / p.H, P1 = p.seg_P - 1;
        const int seqv = (r / P1) * p.seg_P + 1 + r % P1;
        bid = (seqv * p.H + hh) * CPC + k % CPC;
        phi_base = (size_t)idx * D * D;
    }
    const int unit = bid / CPC, jh = bid % CPC, j0 = 64 * jh;
    const int rank = unit / p.H, h = unit % p.H;
    const int seq = p.order ? p.order[rank] : rank;
    long start, len, chunk0;
    if (p.cu_seqlens) {
        start = p.cu_seqlens[seq];
        len = (long)p.cu_seqlens[seq + 1] - start;
        chunk0 = p.chunk_prefix[seq];
    } else if (segP > 1) {   // segment seq % segP of sequence seq / segP
        int tile0, ntiles;
        seg_tiles(p.seg_q, p.seg_r, seq % segP, tile0, ntiles);
        start = (long)(seq / segP) * p.seg_T + 128L * tile0;
        len = 128L * ntiles;
        chunk0 = (long)(seq / segP) * p.seg_nch + 2L * tile0;
    } else {
        start = (long)seq * p.T;
        len = p.T;
        chunk0 = (long)seq * p.nch_fixed;
    }
    const int nch = (int)((len + C - 1) / C);
    const size_t sbase = ((size_t)seq * p.H + h) * D * D;
    // the initial state: S0, zero for a later segment of a split sequence, the
    // identity's columns for a transition pass (s0 == nullptr for the last two)
    const float *s0 = p.S0;
    if (segP > 1)
        s0 = (!phi && p.S0 && seq % segP == 0) ? p.S0 + ((size_t)(seq / segP) * p.H + h) * D * D
                                               : nullptr;
    else if (s0)
        s0 += sbase;
    // In the fused launch the main warps first compute a phase-1 item; the MMA
    // and load warps meanwhile copy the CTA's 64 columns of S0 into shared
    // memory (the S, U and U' operand space, 32 KB, unused until the pass
    // starts) as 16-byte chunk ch of row r at chunk slot ch * 128 + r, which
    // the main warps then read without bank conflicts.
    const bool pre_s0 = kFused && kW == 64 && s0 != nullptr;
    float4 *s0_stage = reinterpret_cast<float4 *>(sm + Cf::SM_S);
    if (pre_s0 && warp >= NMAIN) {
        constexpr int NH = Cf::THREADS - NMAIN * 32;   // the helper threads
#pragma unroll 4
        for (int idx = tid - NMAIN * 32; idx < 2048; idx += NH) {
            const int ch = idx >> 7, r = idx & 127;   // 16 chunks of 16 bytes x 128 rows
            s0_stage[idx] = *reinterpret_cast<const float4 *>(s0 + (size_t)r * D + j0 + 4 * ch);
        }
    }

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_ld[i], 1);
            mbar_init(&bar_empty[i], 2);   // committed by both MMA issuers
        }
        mbar_init(&bar_px, 1);
        mbar_init(&bar_u, NMAIN);    // one arrival per main warp: U' written, S scaled
        mbar_init(&bar_u2, NMAIN);   // one arrival per main warp: U written
        mbar_init(&bar_z, 1);
        mbar_init(&bar_y[0], 1);
        mbar_init(&bar_y[1], 1);
        mbar_init(&bar_s, NMAIN);   // one arrival per main warp
        mbar_init(&bar_fin, 1);
        mbar_init(&bar_fin_y, 1);
        fence_mbar_init();
        // an error already reported: read once, so that the whole CTA
        // agrees (threads reading the word at different times might not)
        sAbort = status_bad(p.status) ? 1 : 0;
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 512);
        tmem_relinquish();
    }
    named_sync(3, Cf::THREADS);
    tc_fence_after();
    const uint32_t tb = tslot;
    if (sAbort) {
        if (warp == 0) tmem_dealloc(tb, 512);
        return;
    }

    auto fail = [&]() {
        *(volatile int *)&sAbort = 1;   // read by the other warps' waits
        set_status(p.status, kDevTimeout);
    };

    if (warp == NMAIN) {
        // ----------------------------------------------------------------- issuer
        const uint32_t id_px = idesc_bf16_f32(128, kW, false, true);
        const uint32_t id_zy = idesc_bf16_f32(128, kW, true, true);
        const uint32_t aS = smem_u32(sS), aU = smem_u32(sU), aUz = smem_u32(sUz);
        int c = 0;
        for (; c < nch; ++c) {
            const int b = c % NS;
            unsigned char *st = sm + b * Cf::ST_BYTES;
            const uint32_t par = (uint32_t)(c & 1), par_st = (uint32_t)((c / NS) & 1);
            // stage landed, and S_c written to shared memory by the main warps
            const bool ok = mbar_wait_or_abort(&bar_ld[b], par_st, &sAbort) &&
                            mbar_wait_or_abort(&bar_s, par, &sAbort);
            if (!__all_sync(0xffffffffu, ok)) { fail(); break; }
            tc_fence_after();
            if (kRecord && p.S_chk && !phi && lane == 0) {
                // S at the chunk's start, for the backward: the bf16 tile as it is
                unsigned char *dst = p.S_chk + ((size_t)(chunk0 + c) * p.H + h) * 32768 + 16384 * jh;
#pragma unroll
                for (int sl = 0; sl < kW / 64; ++sl)
                    bulk_store(dst + 16384 * sl, sS + sl * Cf::S_SLAB, 16384u);
                bulk_commit_group();
            }
            if (lane == 0) {
                const uint32_t aQW = smem_u32(st + ST_QW);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tb + Cf::TM_PX + kW * (c & 1),
                             sdesc_sw128(aQW + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                             sdesc_sw128(aS + ks * 2048, kW == 64 ? 8192 : Cf::S_SLAB, 1024),
                             id_px, ks > 0);
                mma_commit(&bar_px);
            }
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_u, par, &sAbort))) { fail(); break; }
            tc_fence_after();
            // the recorded copy has read S_c before Z lets the main warps overwrite it
            if (kRecord && p.S_chk && !phi && lane == 0) bulk_wait_group_read0();
            if (lane == 0) {
                const uint32_t aKT = smem_u32(st + ST_KT);
                // S_b += K^T U' (S_b, scaled by exp(g_C) by the main warps, is the
                // accumulator): A = K read MN-major (M = dk, two 64-feature blocks)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tb + Cf::TM_S, sdesc_sw128(aKT + ks * 2048, 8192, 1024),
                             sdesc_sw128(aUz + ks * 2048, 8192, 1024), id_zy, 1u);
                mma_commit(&bar_z);
                mma_commit(&bar_empty[b]);   // [X | P] and Z are done with the stage
            }
            __syncwarp();
        }
        // every MMA issued has completed before the CTA releases its TMEM
        if (lane == 0) mma_commit(&bar_fin);
        if (kRecord && p.S_chk && lane == 0) bulk_wait_group0();
        __syncwarp();
        (void)mbar_wait(&bar_fin, 0u);
    } else if (warp == NMAIN + 2) {
        // ----------------------------------------------------------------- Y issue
        // Y = A U once U is written (bar_u2), from a thread of its own: an MMA
        // issue waits for room in the tensor pipe, and the chain's issuer must
        // be free when the next state is published.
        const uint32_t id_zy = idesc_bf16_f32(128, kW, true, true);
        const uint32_t aU = smem_u32(sU);
        for (int c = 0; c < nch; ++c) {
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_u2, (uint32_t)(c & 1), &sAbort))) {
                fail();
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t aA = smem_u32(sm + (c % NS) * Cf::ST_BYTES + ST_A);
                // A read MN-major from A^T; its second 64-row block (rows 64..127
                // of the product, never read) points at U~
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tb + Cf::TM_Y + Cf::Y_STRIDE * (c & 1),
                             sdesc_sw128(aA + ks * 2048, 8192, 1024),
                             sdesc_sw128(aU + ks * 2048, 8192, 1024), id_zy, ks > 0);
                mma_commit(&bar_y[c & 1]);
                mma_commit(&bar_empty[c % NS]);   // Y is done with the stage
            }
            __syncwarp();
        }
        // every MMA of this thread has completed before the CTA releases its TMEM
        if (lane == 0) mma_commit(&bar_fin_y);
        __syncwarp();
        (void)mbar_wait(&bar_fin_y, 0u);
    } else if (warp == NMAIN + 1) {
        // ----------------------------------------------------------------- loads
        // Chunk n goes to stage n % NSTAGE once the products of chunk
        // n - NSTAGE are done with it (bar_empty) and, in the fused launch,
        // once the phase-1 item holding chunk n is published (flag of pair
        // n / 2, counted per unit).
        int n = 0;
        for (; n < nch; ++n) {
            const int b = n % NS, k = n / NS;
            if (k >= 1 &&
                !__all_sync(0xffffffffu,
                            mbar_wait_or_abort(&bar_empty[b], (uint32_t)((k - 1) & 1), &sAbort))) {
                fail();
                break;
            }
            int st = 1;
            if (kFused && lane == 0) {
                const long long t0 = clock64();
                if (n == 0 && p.test_gate != nullptr)
                    while (ld_acquire_u32(p.test_gate) == 0u)
                        if (clock64() - t0 >= p.flag_wait_limit) { st = 0; break; }
                const unsigned *f = p.flags + (long)(n >> 1) * p.n_units + unit;
                while (st && ld_acquire_u32(f) == 0u)
                    if (clock64() - t0 >= p.flag_wait_limit) { st = 0; break; }
            }
            if (!__shfl_sync(0xffffffffu, st, 0)) { fail(); break; }
            if (lane == 0) {
                if (kFused) fence_proxy_async_global();
                const long slot = (chunk0 + n) * p.H + h;
                issue_stage<kW>(sm + b * Cf::ST_BYTES, sG + b * C, &bar_ld[b], mq, mk, mw, mu, ma,
                            p.g_ws + slot * C, h, (int)(start + (long)n * C), (int)slot, j0);
            }
            __syncwarp();
        }
        // on an early exit, the loads still in flight (at most one per stage)
        // land before the CTA leaves
        if (sAbort)
            for (int k = n > NS ? n - NS : 0; k < n; ++k)
                (void)mbar_wait(&bar_ld[k % NS], (uint32_t)((k / NS) & 1));
    } else {
        // ----------------------------------------------------------------- main
        // Thread (L, hf) holds row L of S_b for the tile columns
        // [c0, c0 + 32 NJ) in NJ groups of 32 (group jj: columns cg = c0 + 32 jj,
        // in 64-column slab cg / 64 of the bf16 operands).
        const size_t rs = (size_t)p.H * D;
        float Sr[NJ][32];
        {
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                const int cg = c0 + 32 * jj;
                const float4 *src = reinterpret_cast<const float4 *>(s0 + (size_t)L * D + j0 + cg);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v = pre_s0 ? s0_stage[(cg / 4 + i) * 128 + L]
                                   : s0     ? src[i]
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                    Sr[jj][4 * i] = v.x; Sr[jj][4 * i + 1] = v.y;
                    Sr[jj][4 * i + 2] = v.z; Sr[jj][4 * i + 3] = v.w;
                }
                if (phi) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) Sr[jj][i] = (L == j0 + cg + i) ? 1.f : 0.f;
                }
                // every main warp has read the staged S0 before any overwrites it
                if (pre_s0) named_sync(4, NMAIN * 32);
                st_row_bf16x32(sS + (cg >> 6) * Cf::S_SLAB, L, cg & 63, Sr[jj]);
                tmem_st_f32x32(tb + lane_base + Cf::TM_S + cg, Sr[jj]);
            }
            tmem_st_wait();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_s);
        }
        const bool pwarp = (warp & 2) != 0;    // lanes 64..127: P rows (tokens L - 64)
        for (int c = 0; c < nch; ++c) {
            const int b = c % NS;
            unsigned char *st = sm + b * Cf::ST_BYTES;
            const uint32_t par = (uint32_t)(c & 1), par_st = (uint32_t)((c / NS) & 1);
            const uint32_t tPX = tb + lane_base + Cf::TM_PX + kW * (c & 1);
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_ld[b], par_st, &sAbort))) {
                fail();
                break;
            }
            // what the stage alone gives (g, the decay factors, the U~ words) is
            // read before the wait for the product
            const float *g = sG + b * C;
            const float gC = g[C - 1];
            const float egC = __expf(gC);
            const int nc = (int)min((long)C, len - (long)c * C);
            float egt = 0.f, ft = 0.f;
            // (the wide form, with 576 threads under its register limit, reads its
            // U~ words after the wait)
            constexpr int NPRE = kW == 64 ? NJ : 0;
            uint4 wu[NJ][4];
            if (pwarp) {
                const int t = L - 64;
                ft = __expf(gC - g[t]);
#pragma unroll
                for (int jj = 0; jj < NPRE; ++jj) {
                    const int cg = c0 + 32 * jj;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        wu[jj][k] = *reinterpret_cast<const uint4 *>(
                            st + ST_U + (cg >> 6) * Cf::U_SLAB + sw128_offset(t, (cg & 63) + 8 * k));
                        if (phi) wu[jj][k] = make_uint4(0u, 0u, 0u, 0u);   // U~ = 0 in a transition pass
                    }
                }
            } else {
                egt = __expf(g[L]);
            }
            // ---- S_b <- exp(g_C) S_b in TMEM (row L, the thread's columns), while
            //      [X | P] runs; Z then accumulates into it ----
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                uint32_t r[32];
                tmem_ld32(tb + lane_base + Cf::TM_S + c0 + 32 * jj, r);
                tmem_ld_wait();
                float s[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) s[i] = egC * __uint_as_float(r[i]);
                tmem_st_f32x32(tb + lane_base + Cf::TM_S + c0 + 32 * jj, s);
            }
            tmem_st_wait();
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_px, par, &sAbort))) {
                fail();
                break;
            }
            tc_fence_after();
            if (pwarp) {
                // ---- U = U~_b - P and U' = exp(g_C - g_t) U for token t = L - 64,
                //      the thread's columns ----
                const int t = L - 64;
                // U' (the B operand of the S update) is written and published
                // first; U (for Y) after
                float u[32];            // kW = 64: U of the thread's 32 columns
                uint32_t pu[2][8];      // kW = 128: U in bf16 pairs, two 16-column halves
                if (kW == 64) {
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const int cg = c0 + 32 * jj;
                    uint32_t r[32];
                    tmem_ld32(tPX + cg, r);
                    tmem_ld_wait();
                    float uz[32];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint4 w = wu[jj][k];
                        if (NPRE == 0) {
                            w = *reinterpret_cast<const uint4 *>(
                                st + ST_U + (cg >> 6) * Cf::U_SLAB + sw128_offset(t, (cg & 63) + 8 * k));
                            if (phi) w = make_uint4(0u, 0u, 0u, 0u);
                        }
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            u[8 * k + 2 * e] = bf_lo(ww[e]) - __uint_as_float(r[8 * k + 2 * e]);
                            u[8 * k + 2 * e + 1] =
                                bf_hi(ww[e]) - __uint_as_float(r[8 * k + 2 * e + 1]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) uz[i] = ft * u[i];
                    st_row_bf16x32(sUz + (cg >> 6) * Cf::U_SLAB, t, cg & 63, uz);
                }
                } else {
                    // 16 columns at a time (register pressure of 576 threads)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int cg = c0 + 16 * hh;
                        uint32_t r[16];
                        tmem_ld16(tPX + cg, r);
                        tmem_ld_wait();
                        uint32_t pz[8];
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            uint4 w = *reinterpret_cast<const uint4 *>(
                                st + ST_U + (cg >> 6) * Cf::U_SLAB + sw128_offset(t, (cg & 63) + 8 * k));
                            if (phi) w = make_uint4(0u, 0u, 0u, 0u);
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float u0 = bf_lo(ww[e]) - __uint_as_float(r[8 * k + 2 * e]);
                                const float u1 = bf_hi(ww[e]) - __uint_as_float(r[8 * k + 2 * e + 1]);
                                pu[hh][4 * k + e] = pack_bf2(u0, u1);
                                pz[4 * k + e] = pack_bf2(ft * u0, ft * u1);
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const uint32_t off = sw128_offset(t, (cg & 63) + 8 * k);
                            *reinterpret_cast<uint4 *>(sUz + (cg >> 6) * Cf::U_SLAB + off) =
                                make_uint4(pz[4 * k], pz[4 * k + 1], pz[4 * k + 2], pz[4 * k + 3]);
                        }
                    }
                }
                if (t >= nc) {
                    // rows past the sequence's end: clear this thread's share of
                    // K's row (the next sequence's tokens or zero fill): with two
                    // column groups, features [32 hf, 32 hf + 32) of both slabs;
                    // with four, features [32 (hf % 2), + 32) of slab hf / 2
                    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        if (NCG == 4 && sl != (hf >> 1)) continue;
                        const int f0 = NCG == 4 ? 32 * (hf & 1) : 32 * hf;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<uint4 *>(st + ST_KT + sl * 8192 +
                                                       sw128_offset(t, f0 + 8 * k)) = zero4;
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_u);
                if (kW == 64) {
                    st_row_bf16x32(sU + (c0 >> 6) * Cf::U_SLAB, t, c0 & 63, u);
                } else {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const int cg = c0 + 16 * hh;
                            *reinterpret_cast<uint4 *>(sU + (cg >> 6) * Cf::U_SLAB +
                                                       sw128_offset(t, (cg & 63) + 8 * k)) =
                                make_uint4(pu[hh][4 * k], pu[hh][4 * k + 1], pu[hh][4 * k + 2],
                                           pu[hh][4 * k + 3]);
                        }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_u2);
            } else {
                // every read of this stage by the main warps (and, with one Y
                // buffer, of the previous chunk's Y) and their scaling of S_b
                // precede their bar_u and bar_u2 arrivals, which precede the
                // products that overwrite or accumulate into them
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar_u);
                    mbar_arrive(&bar_u2);
                }
            }

            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_z, par, &sAbort))) { fail(); break; }
            tc_fence_after();
            // ---- S_b = exp(g_C) S_b + Z is complete in TMEM: its bf16 copy for the
            //      next [X | P] (row L, the thread's columns) ----
            if (c + 1 < nch) {
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const int cg = c0 + 32 * jj;
                    uint32_t r[32];
                    tmem_ld32(tb + lane_base + Cf::TM_S + cg, r);
                    tmem_ld_wait();
                    float s[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
                    st_row_bf16x32(sS + (cg >> 6) * Cf::S_SLAB, L, cg & 63, s);
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_s);
            }
            // ---- O_b = diag(exp g) X + Y for token t = L (X rows), after S is published ----
            if (!pwarp) {
                if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&bar_y[c & 1],
                                                                 (uint32_t)((c >> 1) & 1), &sAbort))) {
                    fail();
                    break;
                }
                tc_fence_after();
                // 32 columns at once (kW = 64), or 16 at a time (kW = 128)
                constexpr int OW = kW == 64 ? 32 : 16;
#pragma unroll
                for (int hh = 0; hh < 32 / OW; ++hh) {
                    const int cg = c0 + OW * hh;
                    uint32_t xr[OW], yr[OW];
                    if (OW == 32) {
                        tmem_ld32(tPX + cg, *reinterpret_cast<uint32_t(*)[32]>(xr));
                        tmem_ld32(tb + lane_base + Cf::TM_Y + Cf::Y_STRIDE * (c & 1) + cg,
                                  *reinterpret_cast<uint32_t(*)[32]>(yr));
                    } else {
                        tmem_ld16(tPX + cg, *reinterpret_cast<uint32_t(*)[16]>(xr));
                        tmem_ld16(tb + lane_base + Cf::TM_Y + Cf::Y_STRIDE * (c & 1) + cg,
                                  *reinterpret_cast<uint32_t(*)[16]>(yr));
                    }
                    tmem_ld_wait();
                    if (L < nc && (!kRecord || (phi ? p.o_phi : p.o) != nullptr)) {
                        uint4 *dst = reinterpret_cast<uint4 *>((phi ? p.o_phi : p.o) +
                                                               (size_t)(start + (long)c * C + L) * rs +
                                                               (size_t)h * D + j0 + cg);
#pragma unroll
                        for (int k = 0; k < OW / 8; ++k) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 8 * k + 2 * e;
                                w[e] = pack_bf2(
                                    fmaf(egt, __uint_as_float(xr[i]), __uint_as_float(yr[i])),
                                    fmaf(egt, __uint_as_float(xr[i + 1]), __uint_as_float(yr[i + 1])));
                            }
                            dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                tc_fence_before();
            }
        }
        if (!sAbort && (phi ? p.S_T_phi != nullptr : p.S_T != nullptr)) {
            // the final state (S0 itself when the sequence is empty), from TMEM
            tc_fence_after();
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                uint32_t r[32];
                tmem_ld32(tb + lane_base + Cf::TM_S + c0 + 32 * jj, r);
                tmem_ld_wait();
                float4 *dst = reinterpret_cast<float4 *>(
                    (phi ? p.S_T_phi + phi_base : p.S_T + sbase) + (size_t)L * D + j0 + c0 + 32 * jj);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                         __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
            }
        }
    }
    tc_fence_before();
    named_sync(3, Cf::THREADS);
    if (warp == 0) tmem_dealloc(tb, 512);
}

__global__ void __launch_bounds__(P2_THREADS, 1)
state_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
             const __grid_constant__ CUtensorMap ma, const TcParams p) {
    extern __shared__ unsigned char smraw[];
    state_run<false, true>(&mq, &mk, &mw, &mu, &ma, p, align1024(smraw), (int)blockIdx.x,
                           (int)threadIdx.x);
}

// One CTA per (sequence, head) -- or, with the sequence split, per virtual
// sequence and per transition pass -- carrying all 128 columns of its state.
constexpr int P2W_THREADS = P2Cfg<128>::THREADS;
__global__ void __launch_bounds__(P2W_THREADS, 1)
state_kernel_wide(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
                  const __grid_constant__ CUtensorMap ma, const TcParams p) {
    extern __shared__ unsigned char smraw[];
    state_run<false, true, 128>(&mq, &mk, &mw, &mu, &ma, p, align1024(smraw), (int)blockIdx.x,
                                (int)threadIdx.x);
}

// ===================================================================== fused launch
// Phase 1 and the state pass in one cooperative launch, one CTA per SM: CTAs
// [0, n_state) run the state pass (two per unit); every other CTA runs two
// phase-1 workers over the work items in chunk-pair-major order, so that the
// state pass consumes chunk pairs as they are published instead of waiting
// for the whole of phase 1.  The state-pass CTAs first compute the first two
// chunk pairs of their own unit themselves (CTA 2u pair 0, CTA 2u + 1 pair
// 1), which they would otherwise wait for, and then start the chain; the
// workers take the items from pair 2 on.  Only the consumer waits (bounded),
// and every CTA is resident (cooperative launch), so the hand-offs cannot
// deadlock.
constexpr int FU_THREADS = 2 * P1_THREADS;
static_assert(FU_THREADS >= P2_THREADS, "fused block size");
constexpr uint32_t FU_SMEM = P2_SMEM > 2 * P1_REGION + 1024 ? P2_SMEM : 2 * P1_REGION + 1024;

// kRecord: the call records S and T of every chunk for the backward (and
// may write no outputs); the other instantiations carry no recording code.
template <bool kSplit, bool kRecord>
__global__ void __launch_bounds__(FU_THREADS, 1)
fused_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mw,
             const __grid_constant__ CUtensorMap mu, const __grid_constant__ CUtensorMap ma,
             const TcParams p, long n_pairs, int n_state, int n_phi) {
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = align1024(smraw);
    const int tid = (int)threadIdx.x;
    const long n_items = n_pairs * p.H;
    const int pre = p.nch_fixed >= 4 ? 2 : 1;   // leading chunk pairs done by the state CTAs
    if ((int)blockIdx.x < n_state + n_phi) {
        // state-pass CTAs (then, with the sequence split, transition-pass CTAs,
        // which only consume); two 64-column CTAs per chain: the three load
        // stages they keep in flight do not fit beside a 128-column tile
        const int unit = (int)blockIdx.x >> 1, jh = (int)blockIdx.x & 1;
        if ((int)blockIdx.x < n_state && jh < pre && tid < P1_THREADS)
            intra_run<true, kRecord>(&mq, &mk, &mv, &mw, &mu, p, n_pairs, sm, tid, 1,
                                     (long)jh * p.n_units + unit, n_items);
        if (tid < P2_THREADS)
            state_run<true, kSplit, 64, kRecord>(&mq, &mk, &mw, &mu, &ma, p, sm, (int)blockIdx.x,
                                                 tid);
        return;
    }
    __shared__ int stagger;
    if (tid == 0) stagger = 0;
    __syncthreads();
    const int w = tid / P1_THREADS;
    intra_run<true, kRecord>(&mq, &mk, &mv, &mw, &mu, p, n_pairs, sm + w * P1_REGION,
                             tid % P1_THREADS, 1 + w, (long)pre * p.n_units, 0, &stagger,
                             1 + w);   // items from the shared counter
}

// ===================================================================== varlen prep
// One CTA: validates cu_seqlens, writes the first chunk of every sequence
// (chunk_prefix[N+1]), the first token row and token count of every chunk
// (chunk_tab, so that phase 1 finds a chunk with one load) and a
// longest-first order of the sequences.
constexpr int PREP_THREADS = 1024;

__global__ void __launch_bounds__(PREP_THREADS)
prep_kernel(const int *cu, int N, int total_T, int *chunk_prefix, int *order, int2 *chunk_tab,
            unsigned *status) {
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
    __syncthreads();
    // (first token row, tokens) of every chunk: a warp per sequence, its
    // lanes over the sequence's chunks
    for (int n = warp; n < N; n += PREP_THREADS / 32) {
        const int c0 = chunk_prefix[n], nc = chunk_prefix[n + 1] - c0;
        const int start = cu[n], len = cu[n + 1] - start;
        for (int c = lane; c < nc; c += 32)
            chunk_tab[c0 + c] = make_int2(start + c * C, min(C, len - c * C));
    }
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

// ===================================================================== sequence split
// A fixed-length sequence run as P segments (the state pass of each segment
// has a P times shorter chain).  The forward is linear in (V, S0) jointly, so
// for a later segment s with start state S_s
//   o = o(V, 0) + Q_corr S_s,   S_end = N_s + Phi_s S_s,
// where o(V, 0), N_s are the segment's outputs from a zero state and
// Q_corr = o(0, I), Phi_s = S_T(0, I) those of the transition pass (U~ = 0,
// S0 = I).  The segment start states follow in order from S_1 = S_end of
// segment 0.

// Per (batch, head, CBW columns): S_1 .. S_{P-1} into Sst (bf16, the
// correction's operand) and S_P as S_T.  The columns are independent.  Each
// thread owns NX columns of one row; Phi_{s+1} and N_{s+1} are fetched into
// registers while the product of segment s runs, and the shared-memory rows
// are float4-aligned (Phi rows of D + 4 floats, S rows of CBW + 4).
constexpr int CB_THREADS = 256;
constexpr int CBW = 16;   // state columns per CTA (two threads per row, CBW / 2 each)
constexpr int CB_PH = D + 4, CB_SS = CBW + 4;
constexpr size_t CB_SMEM = ((size_t)D * CB_PH + (size_t)D * CB_SS) * sizeof(float);

__global__ void __launch_bounds__(CB_THREADS)
split_combine_kernel(const float *__restrict__ Nbuf, const float *__restrict__ Phi,
                     __nv_bfloat16 *__restrict__ Sst, float *__restrict__ S_T, int H, int P,
                     const unsigned *status) {
    extern __shared__ float cb_sm[];
    constexpr int NX = CBW / 2;
    constexpr int NV = D * D / 4 / CB_THREADS;   // float4 of Phi per thread
    float(*Ph)[CB_PH] = reinterpret_cast<float(*)[CB_PH]>(cb_sm);                       // Phi_s
    float(*Ss)[CB_SS] = reinterpret_cast<float(*)[CB_SS]>(cb_sm + (size_t)D * CB_PH);   // S_s
    if (status_bad(status)) return;
    const int unit = blockIdx.x, b = unit / H, h = unit % H, jb = blockIdx.y * CBW;
    const int tid = threadIdx.x, i = tid >> 1, j0 = (tid & 1) * NX;
    auto n_block = [&](int sg) {   // row i, columns jb + j0 .. of N_sg
        return reinterpret_cast<const float4 *>(Nbuf + ((size_t)(b * P + sg) * H + h) * D * D +
                                                (size_t)i * D + jb + j0);
    };
    auto phi_of = [&](int sg) {    // Phi of segment sg >= 1
        return reinterpret_cast<const float4 *>(Phi + ((size_t)(b * (P - 1) + sg - 1) * H + h) * D * D);
    };
    float cur[NX], nx[NX];
    float4 buf[NV];
    {
        const float4 *n0 = n_block(0);
        const float4 a0 = n0[0], a1 = n0[1];
        cur[0] = a0.x; cur[1] = a0.y; cur[2] = a0.z; cur[3] = a0.w;
        cur[4] = a1.x; cur[5] = a1.y; cur[6] = a1.z; cur[7] = a1.w;
    }
    if (P > 1) {
        const float4 *src = phi_of(1);
#pragma unroll
        for (int n = 0; n < NV; ++n) buf[n] = src[tid + n * CB_THREADS];
        const float4 *n1 = n_block(1);
        const float4 a0 = n1[0], a1 = n1[1];
        nx[0] = a0.x; nx[1] = a0.y; nx[2] = a0.z; nx[3] = a0.w;
        nx[4] = a1.x; nx[5] = a1.y; nx[6] = a1.z; nx[7] = a1.w;
#pragma unroll
        for (int n = 0; n < NV; ++n) {
            const int e = (tid + n * CB_THREADS) * 4;
            *reinterpret_cast<float4 *>(&Ph[e / D][e % D]) = buf[n];
        }
    }
    for (int sg = 1; sg < P; ++sg) {
        // S_sg: the correction's operand (bf16), and the product's right factor
        __nv_bfloat16 *dst = Sst + ((size_t)(b * (P - 1) + sg - 1) * H + h) * D * D +
                             (size_t)i * D + jb + j0;
        uint4 pk;
        pk.x = pack_bf2(cur[0], cur[1]); pk.y = pack_bf2(cur[2], cur[3]);
        pk.z = pack_bf2(cur[4], cur[5]); pk.w = pack_bf2(cur[6], cur[7]);
        *reinterpret_cast<uint4 *>(dst) = pk;
        *reinterpret_cast<float4 *>(&Ss[i][j0]) = make_float4(cur[0], cur[1], cur[2], cur[3]);
        *reinterpret_cast<float4 *>(&Ss[i][j0 + 4]) = make_float4(cur[4], cur[5], cur[6], cur[7]);
        __syncthreads();   // Ss written; Ph holds Phi_sg
        const bool more = sg + 1 < P;
        float nn[NX];
        if (more) {        // the next segment's Phi and N, in flight during the product
            const float4 *src = phi_of(sg + 1);
#pragma unroll
            for (int n = 0; n < NV; ++n) buf[n] = src[tid + n * CB_THREADS];
            const float4 *nb = n_block(sg + 1);
            const float4 a0 = nb[0], a1 = nb[1];
            nn[0] = a0.x; nn[1] = a0.y; nn[2] = a0.z; nn[3] = a0.w;
            nn[4] = a1.x; nn[5] = a1.y; nn[6] = a1.z; nn[7] = a1.w;
        }
#pragma unroll
        for (int x = 0; x < NX; ++x) cur[x] = nx[x];
#pragma unroll 2
        for (int k4 = 0; k4 < D; k4 += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(&Ph[i][k4]);
            const float fk[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 s0 = *reinterpret_cast<const float4 *>(&Ss[k4 + e][j0]);
                const float4 s1 = *reinterpret_cast<const float4 *>(&Ss[k4 + e][j0 + 4]);
                cur[0] = fmaf(fk[e], s0.x, cur[0]); cur[1] = fmaf(fk[e], s0.y, cur[1]);
                cur[2] = fmaf(fk[e], s0.z, cur[2]); cur[3] = fmaf(fk[e], s0.w, cur[3]);
                cur[4] = fmaf(fk[e], s1.x, cur[4]); cur[5] = fmaf(fk[e], s1.y, cur[5]);
                cur[6] = fmaf(fk[e], s1.z, cur[6]); cur[7] = fmaf(fk[e], s1.w, cur[7]);
            }
        }
        __syncthreads();   // Ph and Ss are no longer read
        if (more) {
#pragma unroll
            for (int x = 0; x < NX; ++x) nx[x] = nn[x];
#pragma unroll
            for (int n = 0; n < NV; ++n) {
                const int e = (tid + n * CB_THREADS) * 4;
                *reinterpret_cast<float4 *>(&Ph[e / D][e % D]) = buf[n];
            }
        }
    }
    if (S_T) {
        float4 *dst = reinterpret_cast<float4 *>(S_T + ((size_t)unit * D + i) * D + jb + j0);
        dst[0] = make_float4(cur[0], cur[1], cur[2], cur[3]);
        dst[1] = make_float4(cur[4], cur[5], cur[6], cur[7]);
    }
}

// o[rows] += Q_corr[rows] S_s for the 128-row tiles of the later segments:
// per tile one tcgen05 MMA chain (M = 128 tokens, N = 128, K = 128), A =
// Q_corr rows (K-major, TMA), B = S_s in bf16 (MN-major, TMA), o rows loaded
// by TMA, added to in shared memory and stored by TMA.  Persistent: CTA i
// takes a contiguous run of tiles (tiles in (batch, head, tile) order, so a
// run shares S_s for many tiles and reloads it only when the segment
// changes); the next tile's Q_corr rows (and S_s) load while this tile's sum
// is formed, its o rows once this tile's store has read shared memory.
constexpr int CR_THREADS = 128;
constexpr uint32_t CR_A = 0, CR_B = 32768, CR_O = 65536, CR_SMEM = 98304 + 1024;

struct CrTile {
    int h, row0, srow;
};

__device__ __forceinline__ CrTile cr_tile(long x, int H, int T, int P, int seg_q, int seg_r,
                                          int later_tiles) {
    const int tau = (int)(x % later_tiles);
    x /= later_tiles;
    const int h = (int)(x % H);
    const long b = x / H;
    int t0, n0;
    seg_tiles(seg_q, seg_r, 0, t0, n0);
    const int j = n0 + tau;   // tile of the sequence, and its segment
    const int sg = j < seg_r * (seg_q + 1) ? j / (seg_q + 1) : seg_r + (j - seg_r * (seg_q + 1)) / seg_q;
    CrTile c;
    c.h = h;
    c.row0 = (int)(b * T + 128L * j);
    c.srow = (int)(((b * (P - 1) + sg - 1) * H + h) * D);   // first row of S_s (bf16 array)
    return c;
}

__global__ void __launch_bounds__(CR_THREADS)
split_correct_kernel(const __grid_constant__ CUtensorMap mqc, const __grid_constant__ CUtensorMap mo,
                     const __grid_constant__ CUtensorMap mss, int H, int T, int P, int seg_q,
                     int seg_r, int later_tiles, long n_tiles, unsigned *status) {
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = align1024(smraw);
    __shared__ uint64_t bar_a, bar_o, bar_b, bar_mma;
    __shared__ uint32_t tslot;
    __shared__ int sok;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (status_bad(status)) return;
    const long x0 = (long)blockIdx.x * n_tiles / gridDim.x;
    const long x1 = (long)(blockIdx.x + 1) * n_tiles / gridDim.x;
    if (x0 >= x1) return;
    if (tid == 0) {
        mbar_init(&bar_a, 1);
        mbar_init(&bar_o, 1);
        mbar_init(&bar_b, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        sok = 1;
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 128);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tslot;
    auto load_rows = [&](const CUtensorMap *m, unsigned char *dst, uint64_t *bar, const CrTile &c) {
        mbar_expect_tx(bar, 32768u);
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                tma_load_3d(dst + sl * 16384 + hf * 8192, m, bar, 64 * sl, c.h, c.row0 + 64 * hf);
    };
    auto load_s = [&](int srow) {
        mbar_expect_tx(&bar_b, 32768u);
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) tma_load_2d(sm + CR_B + nb * 16384, &mss, &bar_b, 64 * nb, srow);
    };
    // thread 0's bookkeeping: loads issued per barrier (phase parities) and
    // the S_s rows in shared memory
    uint32_t n_a = 0, n_o = 0, n_b = 0, n_mma = 0;
    int cur_srow = -1;
    if (tid == 0) {
        const CrTile c = cr_tile(x0, H, T, P, seg_q, seg_r, later_tiles);
        load_s(c.srow);
        cur_srow = c.srow;
        ++n_b;
        load_rows(&mqc, sm + CR_A, &bar_a, c);
        ++n_a;
        load_rows(&mo, sm + CR_O, &bar_o, c);
        ++n_o;
    }
    for (long x = x0; x < x1; ++x) {
        const CrTile c = cr_tile(x, H, T, P, seg_q, seg_r, later_tiles);
        if (tid == 0) {
            // this tile's S_s (the last one loaded) and Q_corr rows
            bool ok = mbar_wait(&bar_b, (n_b - 1) & 1u) && mbar_wait(&bar_a, (n_a - 1) & 1u);
            if (ok) {
                tc_fence_after();
                const uint32_t aA = smem_u32(sm + CR_A), aB = smem_u32(sm + CR_B);
                const uint32_t id = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tb, sdesc_sw128(aA + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                             sdesc_sw128(aB + ks * 2048, 16384, 1024), id, ks > 0);
                mma_commit(&bar_mma);
                ++n_mma;
                ok = mbar_wait(&bar_mma, (n_mma - 1) & 1u);
                if (!ok) (void)mbar_wait(&bar_mma, (n_mma - 1) & 1u);   // done before TMEM is reused
            }
            if (ok && x + 1 < x1) {   // A and B are free: the next tile's operands
                const CrTile cn = cr_tile(x + 1, H, T, P, seg_q, seg_r, later_tiles);
                if (cn.srow != cur_srow) {
                    load_s(cn.srow);
                    cur_srow = cn.srow;
                    ++n_b;
                }
                load_rows(&mqc, sm + CR_A, &bar_a, cn);
                ++n_a;
            }
            if (ok) ok = mbar_wait(&bar_o, (n_o - 1) & 1u);
            if (!ok) {
                sok = 0;
                set_status(status, kDevTimeout);
            }
        }
        __syncthreads();
        if (!sok) break;
        tc_fence_after();
        {
            const int rrow = warp * 32 + lane;
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t rr[32];
                tmem_ld32(tb + ((uint32_t)(warp * 32) << 16) + c4 * 32, rr);
                tmem_ld_wait();
                unsigned char *tile = sm + CR_O + (c4 >> 1) * 16384;
                const int col0 = (32 * c4) & 63;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint4 *pk = reinterpret_cast<uint4 *>(tile + sw128_offset(rrow, col0 + 8 * k));
                    const uint4 v = *pk;
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t o4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o4[e] = pack_bf2(bf_lo(w[e]) + __uint_as_float(rr[8 * k + 2 * e]),
                                         bf_hi(w[e]) + __uint_as_float(rr[8 * k + 2 * e + 1]));
                    *pk = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();   // the sum is in shared memory; TMEM is free for the next product
        if (tid == 0) {
#pragma unroll
            for (int sl = 0; sl < 2; ++sl)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    tma_store_3d(&mo, sm + CR_O + sl * 16384 + hf * 8192, 64 * sl, c.h, c.row0 + 64 * hf);
            bulk_commit_group();
            if (x + 1 < x1) {   // the next tile's o rows once the store has read these
                bulk_wait_group_read0();
                load_rows(&mo, sm + CR_O, &bar_o,
                          cr_tile(x + 1, H, T, P, seg_q, seg_r, later_tiles));
                ++n_o;
            }
        }
    }
    if (tid == 0) {
        bulk_wait_group0();   // every store complete before the CTA leaves
        if (!sok) {           // loads still in flight land before shared memory is released
            if (n_a) (void)mbar_wait(&bar_a, (n_a - 1) & 1u);
            if (n_o) (void)mbar_wait(&bar_o, (n_o - 1) & 1u);
            if (n_b) (void)mbar_wait(&bar_b, (n_b - 1) & 1u);
        }
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 128);
}

// ===================================================================== host side
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
    size_t meta, g, W, U, A, total;
};

// Offset (in ints) of the varlen chunk table in the meta area: after the
// chunk prefix [N + 1] and the order [N], on an 8-byte boundary.
size_t tab_offset(int n_seq) { return ((size_t)2 * n_seq + 1 + 1) & ~(size_t)1; }

WsLayout layout(long n_chunks, int H, int n_seq) {
    const size_t slots = (size_t)n_chunks * H;
    // meta: the varlen chunk prefix, order and chunk table (from an 8-byte
    // boundary, one entry per chunk slot and one past), or the fused
    // launch's ready flags
    const size_t meta_ints = std::max(tab_offset(n_seq) + 2 * ((size_t)n_chunks + 1),
                                      (size_t)((n_chunks + 1) / 2) * H + 1);
    WsLayout L;
    L.meta = 0;
    L.g = align_up(meta_ints * sizeof(int), 1024);
    L.W = L.g + align_up(slots * C * sizeof(float), 1024);
    L.U = L.W + slots * C * D * 2;
    L.A = L.U + slots * C * D * 2;
    L.total = L.A + slots * C * C * 2;
    return L;
}

// Chains of a sequence split into P segments: P state passes and P - 1
// transition passes per (sequence, head).
long split_chains(long units, int P) { return units * P + units * (P - 1); }

// Sequence split factor P for a fixed-length batch (1: none).  The sequence
// is cut into P segments of whole 128-token tiles, as equal as the tile count
// allows (the first ones one tile longer).  A P is eligible if its state and
// transition passes fit on the SMs at once, as two 64-column CTAs per chain
// with segments of at least 1024 tokens, or as one 128-column CTA per chain
// (a pass with two load stages, which pays only on long chains) with
// segments of at least 4096 tokens; of the eligible P <= 8 (and no split)
// the one with the shortest longest chain is taken, weighing a 128-column
// chain step as 3/2 of a 64-column one -- few heads and long sequences, where
// the serial chain of the state pass dominates.  The environment variable
// KLA_SEQ_SPLIT=P sets it (any P up to the tile count; KLA_SEQ_SPLIT=1
// disables the split).
int split_factor(int n_seq, int T, int H, bool varlen) {
    if (varlen || T <= 0 || T % 128 != 0) return 1;
    const int tiles = T / 128;
    auto valid = [&](int P) { return P >= 2 && P <= tiles; };
    if (const char *e = getenv("KLA_SEQ_SPLIT")) {
        const int P = atoi(e);
        return valid(P) ? P : 1;
    }
    const long units = (long)n_seq * H, sms = sm_count();
    // chain cost in half-steps: a 64-column chain step counts 2, a 128-column
    // one 3 (measured about 1.4 and 2.1 us per chunk)
    long best_cost = (long)(T / C) * (2 * units <= sms ? 2 : 3);
    int best = 1;
    for (int P = 2; P <= 8 && P <= tiles; ++P) {
        const int shortest = tiles / P, longest = (tiles + P - 1) / P;
        long cost = -1;
        if (shortest * 128 >= 1024 && 2 * split_chains(units, P) <= sms)
            cost = 2L * 2 * longest;
        else if (shortest * 128 >= 4096 && split_chains(units, P) <= sms)
            cost = 3L * 2 * longest;
        if (cost >= 0 && cost < best_cost) {
            best_cost = cost;
            best = P;
        }
    }
    return best;
}

// A split whose chains in two 64-column CTAs each would outnumber the SMs
// runs them as one 128-column CTA each (two launches).
bool split_wide(long units, int P) { return P > 1 && 2 * split_chains(units, P) > sm_count(); }

struct SplitLayout {
    size_t N, Phi, Qc, Sst, total;
};

// After the chunk workspace: N (the end states of every segment from its own
// start, fp32), Phi (segments >= 1, fp32), Q_corr rows ([total_T][H][128]
// bf16), the segment start states S_1.. in bf16.
SplitLayout split_layout(int n_seq, int T, int H, int P) {
    SplitLayout L{};
    if (P <= 1) return L;
    const size_t dd = (size_t)D * D;
    L.N = 0;
    L.Phi = L.N + (size_t)n_seq * P * H * dd * 4;
    L.Qc = L.Phi + (size_t)n_seq * (P - 1) * H * dd * 4;
    L.Sst = L.Qc + align_up((size_t)n_seq * T * H * D * 2, 1024);
    L.total = L.Sst + (size_t)n_seq * (P - 1) * H * dd * 2;
    return L;
}

// The fused launch serves fixed-length batches with an even number of chunks
// per (virtual) sequence, equal segments when split, whose state pass (with
// the sequence split: state and transition passes) fits on at most half of
// the SMs; with fewer SMs left to
// phase 1 its items arrive more slowly than the chain consumes them.
bool use_fused(const Problem &p) {
    if (p.cu_seqlens != nullptr || p.T <= 0) return false;
    // a call recording the chunk-start states for the backward does not split
    const int P = p.S_chk ? 1 : split_factor(p.n_seq, p.T, p.H, false);
    if (P > 1 && p.T % (P * 128) != 0) return false;   // segments of unequal length
    const int nch = (p.T / P + C - 1) / C;
    if (nch % 2 != 0) return false;
    return 2 * split_chains((long)p.n_seq * p.H, P) <= sm_count() / 2;
}

// The two-launch state pass runs one 128-column CTA per (sequence, head)
// where two 64-column CTAs per head would not all be resident at once (more
// than one CTA per SM, so the pass is bound by how many chains run side by
// side, not by the length of one); the sequence split keeps the narrow pass.
// KLA_WIDE_STATE=0 / 1 forces either form.
bool use_wide_state(long n_units, int P) {
    if (P > 1) return false;
    if (const char *e = getenv("KLA_WIDE_STATE")) return atoi(e) != 0;
    return 2 * n_units > sm_count();
}

}  // namespace

bool chunk_tc_supported(int d, int dtype) { return d == 128 && dtype == 1; }

size_t chunk_tc_reset_bytes(const Problem &p, long n_chunks_upper) {
    // the ready flags and the work-item counter after them
    return use_fused(p) ? ((size_t)((n_chunks_upper + 1) / 2) * p.H + 1) * sizeof(unsigned) : 0;
}

size_t chunk_tc_workspace_bytes(long n_chunks_upper, int H, int n_seq) {
    return layout(n_chunks_upper, H, n_seq).total;
}

void chunk_tc_ws_views(void *ws, long n_chunks_upper, int H, int n_seq, float **g, void **W,
                       void **A) {
    const WsLayout L = layout(n_chunks_upper, H, n_seq);
    unsigned char *b = static_cast<unsigned char *>(ws);
    *g = reinterpret_cast<float *>(b + L.g);
    *W = b + L.W;
    *A = b + L.A;
}

size_t chunk_tc_split_bytes(int n_seq, int T, int H) {
    const int P = split_factor(n_seq, T, H, false);
    if (P <= 1) return 0;
    // the chunk workspace of the P-times-more virtual sequences, then the split buffers
    const long n_chunks = (long)n_seq * ((T + C - 1) / C);
    const size_t base = align_up(layout(n_chunks, H, n_seq * P).total, 1024);
    return base + split_layout(n_seq, T, H, P).total - layout(n_chunks, H, n_seq).total;
}

cudaError_t launch_split_tail(const Problem &p0, const Problem &p, const TcParams &tp, int P,
                              unsigned char *sws, const SplitLayout &SL, cudaStream_t s);

cudaError_t launch_chunk_tc(const Problem &p0, long n_chunks_upper, cudaStream_t s) {
    if (p0.n_seq == 0) return cudaSuccess;
    // the kernels index work items and chunk slots in 32 bits
    if (n_chunks_upper > INT32_MAX || (n_chunks_upper + 1) / 2 * (long)p0.H > INT32_MAX)
        return cudaErrorInvalidValue;
    if (tmap::encode_fn() == nullptr) return cudaErrorNotSupported;
    // a split sequence runs as P virtual sequences (its segments: same rows,
    // same chunk slots); p keeps the virtual count, and T / P as the segment
    // length of an equal split (the fused launch's item order)
    const bool record = p0.S_chk != nullptr;   // backward recording: no split
    const int P = !record ? split_factor(p0.n_seq, p0.T, p0.H, p0.cu_seqlens != nullptr) : 1;
    Problem p = p0;
    if (P > 1) {
        p.n_seq = p0.n_seq * P;
        p.T = p0.T / P;
    }
    const WsLayout L = layout(n_chunks_upper, p.H, p.n_seq);
    unsigned char *ws = static_cast<unsigned char *>(p.ws);
    const size_t split_base = align_up(L.total, 1024);
    const SplitLayout SL = split_layout(p0.n_seq, p0.T, p0.H, P);
    if (p.ws_bytes < (P > 1 ? split_base + SL.total : L.total)) return cudaErrorInvalidValue;

    TcParams tp{};
    tp.H = p.H;
    tp.n_seq = p.n_seq;
    tp.T = p.T;
    tp.total_T = p.total_T;
    tp.nch_fixed = p.cu_seqlens ? 0 : (p.T + C - 1) / C;
    tp.eps = p.eps;
    tp.beta_mode = p.beta_mode;
    tp.seg_P = P;
    if (P > 1) {
        tp.seg_T = p0.T;
        tp.seg_nch = p0.T / C;
        tp.seg_q = p0.T / 128 / P;
        tp.seg_r = p0.T / 128 % P;
    }
    tp.alpha = p.alpha;
    tp.eta = p.eta;
    tp.S0 = p.S0;
    tp.S_T = p.S_T;
    const bool fused = use_fused(p0);
    bool wide_split = !fused && split_wide((long)p0.n_seq * p0.H, P);
    if (P > 1 && !fused) {
        // phase 1 of the two-launch path runs over the real sequences (the
        // chunk slots are the same); only the state pass sees the segments
        tp.n_seq = p0.n_seq;
        tp.T = p0.T;
        tp.nch_fixed = p0.T / C;
    }
    if (P > 1) {   // the virtual sequences' end states go to N, not to S_T
        tp.S_T = reinterpret_cast<float *>(ws + split_base + SL.N);
        tp.phi_first = (wide_split ? 1 : 2) * p.n_seq * p.H;
        tp.o_phi = reinterpret_cast<__nv_bfloat16 *>(ws + split_base + SL.Qc);
        tp.S_T_phi = reinterpret_cast<float *>(ws + split_base + SL.Phi);
    }
    tp.o = static_cast<__nv_bfloat16 *>(p.o);
    tp.cu_seqlens = p.cu_seqlens;
    tp.status = p.status;
    tp.g_ws = reinterpret_cast<float *>(ws + L.g);
    tp.W_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.W);
    tp.U_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.U);
    tp.A_ws = reinterpret_cast<__nv_bfloat16 *>(ws + L.A);
    int *chunk_prefix = reinterpret_cast<int *>(ws + L.meta);
    int *order = chunk_prefix + p.n_seq + 1;
    int2 *chunk_tab = reinterpret_cast<int2 *>(chunk_prefix + tab_offset(p.n_seq));
    tp.chunk_prefix = p.cu_seqlens ? chunk_prefix : nullptr;
    tp.order = p.cu_seqlens ? order : nullptr;
    tp.chunk_tab = p.cu_seqlens ? chunk_tab : nullptr;

    CUtensorMap mq, mk, mv, mw, mu, ma;
    const long slots = n_chunks_upper * p.H;
    if (!tmap::rows_3d(&mq, p.q, p.H, p.total_T, C) || !tmap::rows_3d(&mk, p.k, p.H, p.total_T, C) ||
        !tmap::rows_3d(&mv, p.v, p.H, p.total_T, C) ||
        !tmap::plain_2d(&mw, tp.W_ws, D, slots * C, C) ||
        !tmap::plain_2d(&mu, tp.U_ws, D, slots * C, C) ||
        !tmap::plain_2d(&ma, tp.A_ws, C, slots * C, C))
        return cudaErrorInvalidValue;

    cudaError_t e;
    if (p.cu_seqlens) {
        prep_kernel<<<1, PREP_THREADS, 0, s>>>(p.cu_seqlens, p.n_seq, p.total_T, chunk_prefix,
                                               order, chunk_tab, p.status);
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
        if ((e = cudaFuncSetAttribute(state_kernel_wide,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)P2Cfg<128>::SMEM)) != cudaSuccess)
            return e;
        attrs = true;
    }
    const long n_pairs = (n_chunks_upper + 1) / 2;
    const long n_items = n_pairs * p.H;
    tp.S_chk = static_cast<unsigned char *>(p0.S_chk);
    tp.T_chk = static_cast<__nv_bfloat16 *>(p0.T_chk);
    if (fused) {
        static bool fattr = false;
        if (!fattr) {
            if ((e = cudaFuncSetAttribute(fused_kernel<false, false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)FU_SMEM)) != cudaSuccess ||
                (e = cudaFuncSetAttribute(fused_kernel<true, false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)FU_SMEM)) != cudaSuccess ||
                (e = cudaFuncSetAttribute(fused_kernel<false, true>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)FU_SMEM)) != cudaSuccess)
                return e;
            fattr = true;
        }
        tp.flags = reinterpret_cast<unsigned *>(ws + L.meta);   // zeroed with the status word
        tp.n_units = p.n_seq * p.H;
        // Test hook: KLA_TEST_FLAG_WAIT=<cycles> bounds every flag wait by
        // that many cycles and makes the state pass first wait on a header
        // word that nothing sets (zeroed with the status word), so that the
        // wait runs out and the timeout path runs.
        tp.flag_wait_limit = kWaitLimitCycles;
        tp.test_gate = nullptr;
        if (const char *e = getenv("KLA_TEST_FLAG_WAIT")) {
            tp.flag_wait_limit = std::max(0LL, atoll(e));
            tp.test_gate = p.status + 1;
        }
        const int n_state = 2 * p.n_seq * p.H;
        const int n_phi = P > 1 ? 2 * p0.n_seq * (P - 1) * p.H : 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)sm_count());
        cfg.blockDim = dim3(FU_THREADS);
        cfg.dynamicSmemBytes = FU_SMEM;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = record  ? cudaLaunchKernelEx(&cfg, fused_kernel<false, true>, mq, mk, mv, mw, mu, ma,
                                         tp, n_pairs, n_state, n_phi)
            : P > 1 ? cudaLaunchKernelEx(&cfg, fused_kernel<true, false>, mq, mk, mv, mw, mu, ma,
                                         tp, n_pairs, n_state, n_phi)
                    : cudaLaunchKernelEx(&cfg, fused_kernel<false, false>, mq, mk, mv, mw, mu, ma,
                                         tp, n_pairs, n_state, n_phi);
        if (e == cudaSuccess) {
            note_launch();
            if (P == 1) return cudaSuccess;
            return launch_split_tail(p0, p, tp, P, ws + split_base, SL, s);
        }
        // not every CTA could be resident (the device is shared or smaller):
        // the two-launch path below needs no co-residency
        (void)cudaGetLastError();
        tp.flags = nullptr;
        tp.n_units = 0;
        wide_split = split_wide((long)p0.n_seq * p0.H, P);
        if (P > 1) tp.phi_first = (wide_split ? 1 : 2) * p.n_seq * p.H;
    }
    const long grid1 = n_items < 2L * sm_count() ? n_items : 2L * sm_count();
    intra_kernel<<<(unsigned)grid1, P1_THREADS, P1_SMEM, s>>>(mq, mk, mv, mw, mu, tp, n_pairs);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long n_phi = P > 1 ? (long)p0.n_seq * (P - 1) * p.H : 0;   // transition chains
    const long n_units = (long)p.n_seq * p.H;
    if (wide_split || use_wide_state(n_units, P))
        state_kernel_wide<<<(unsigned)(n_units + n_phi), P2W_THREADS, P2Cfg<128>::SMEM, s>>>(
            mq, mk, mw, mu, ma, tp);
    else
        state_kernel<<<(unsigned)(2 * (n_units + n_phi)), P2_THREADS, P2_SMEM, s>>>(mq, mk, mw, mu,
                                                                                  ma, tp);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess || P == 1) return e;
    return launch_split_tail(p0, p, tp, P, ws + split_base, SL, s);
}

// Split: the segment start states, then the corrections of the later segments.
cudaError_t launch_split_tail(const Problem &p0, const Problem &p, const TcParams &tp, int P,
                              unsigned char *sws, const SplitLayout &SL, cudaStream_t s) {
    cudaError_t e;
    __nv_bfloat16 *Sst = reinterpret_cast<__nv_bfloat16 *>(sws + SL.Sst);
    static bool battr = false;
    if (!battr) {
        if ((e = cudaFuncSetAttribute(split_combine_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)CB_SMEM)) != cudaSuccess)
            return e;
        battr = true;
    }
    split_combine_kernel<<<dim3((unsigned)(p0.n_seq * p0.H), D / CBW), CB_THREADS, CB_SMEM, s>>>(
        tp.S_T, tp.S_T_phi, Sst, p0.S_T, p0.H, P, p0.status);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    CUtensorMap mqc, mo, mss;
    if (!tmap::rows_3d(&mqc, tp.o_phi, p.H, p.total_T, C) ||
        !tmap::rows_3d(&mo, p0.o, p.H, p.total_T, C) ||
        !tmap::plain_2d(&mss, Sst, D, (long)p0.n_seq * (P - 1) * p.H * D, 128))
        return cudaErrorInvalidValue;
    static bool cattr = false;
    if (!cattr) {
        if ((e = cudaFuncSetAttribute(split_correct_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)CR_SMEM)) != cudaSuccess)
            return e;
        cattr = true;
    }
    int t0, n0;
    seg_tiles(tp.seg_q, tp.seg_r, 0, t0, n0);
    const int later_tiles = p0.T / 128 - n0;
    const long n_tiles = (long)p0.n_seq * p.H * later_tiles;
    const long grid = std::min<long>(n_tiles, 2L * sm_count());   // two CTAs per SM
    split_correct_kernel<<<(unsigned)grid, CR_THREADS, CR_SMEM, s>>>(
        mqc, mo, mss, p.H, p0.T, P, tp.seg_q, tp.seg_r, later_tiles, n_tiles, p0.status);
    note_launch();
    return cudaGetLastError();
}

}  // namespace kla
