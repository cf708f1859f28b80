// Inverse of a unit lower-triangular 64 x 64 matrix on the CUDA cores, for
// the chunk solver T = (I + A)^{-1} (A strictly lower triangular) of the
// CUDA-core kernels.
#pragma once

namespace kla {

// T = (I + A)^{-1} by blocks: the four diagonal 16 x 16 blocks by forward
// substitution (64 threads, one column each), then twice the merge
//   [[D1, 0], [L21, D2]]^{-1} = [[D1^{-1}, 0], [-D2^{-1} L21 D1^{-1}, D2^{-1}]]
// (32 x 32 blocks from pairs of 16 x 16, then the whole 64 x 64), whose two
// products use all 256 threads.  A and T are 64-row arrays with padded rows
// of LA and LT floats; scratch holds 32 x 33 floats.  Every thread of the
// 256-thread block calls it; it ends with a barrier.
template <int LA, int LT>
__device__ inline void invert_unit_lower64(const float (*A)[LA], float (*Tm)[LT], float *scratch,
                                           int tid) {
    for (int x = tid; x < 64 * 64; x += 256) {
        const int t = x >> 6, s = x & 63;
        if ((t >> 4) != (s >> 4)) Tm[t][s] = 0.f;
    }
    if (tid < 64) {
        const int o = (tid >> 4) * 16, c = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float a = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < r; ++s) a = fmaf(-A[o + r][o + s], x[s], a);
            x[r] = a;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tm[o + r][o + c] = x[r];
    }
    __syncthreads();
    {   // 32 x 32: Y = L21 D1 for both pairs (p = tid / 128), two columns per thread
        float(*Y)[17] = reinterpret_cast<float(*)[17]>(scratch);   // [2 * 16][17]
        const int p = tid >> 7, r = (tid >> 3) & 15, c0 = (tid & 7) * 2, o = 32 * p;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int c = c0 + cc;
            float y = 0.f;
            for (int s = c; s < 16; ++s) y = fmaf(A[o + 16 + r][o + s], Tm[o + s][o + c], y);
            Y[16 * p + r][c] = y;
        }
        __syncthreads();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int c = c0 + cc;
            float x = 0.f;
            for (int s = 0; s <= r; ++s) x = fmaf(Tm[o + 16 + r][o + 16 + s], Y[16 * p + s][c], x);
            Tm[o + 16 + r][o + c] = -x;
        }
        __syncthreads();
    }
    {   // 64 x 64: Y = L21 D1 with 32 x 32 blocks, four columns per thread
        float(*Y)[33] = reinterpret_cast<float(*)[33]>(scratch);   // [32][33]
        const int r = tid >> 3, c0 = tid & 7;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = c0 + 8 * k;
            float y = 0.f;
            for (int s = c; s < 32; ++s) y = fmaf(A[32 + r][s], Tm[s][c], y);
            Y[r][c] = y;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = c0 + 8 * k;
            float x = 0.f;
            for (int s = 0; s <= r; ++s) x = fmaf(Tm[32 + r][32 + s], Y[s][c], x);
            Tm[32 + r][c] = -x;
        }
        __syncthreads();
    }
}

}  // namespace kla
