// Shared-memory tile loads for the CUDA-core chunk kernels.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace kla {

__device__ __forceinline__ void unpack16(const uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4 v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}

// Rows 0 .. ROWS-1 of a token-major tensor (token row r, head h at element
// (r * H + h) * ld), columns col0 .. col0 + W - 1, into the fp32 tile dst
// (row stride LDS floats); rows >= nc are zero.  16-byte loads (8 bf16 or 4
// fp32 values), all issued before the first store.  The source row offsets
// must be 16-byte aligned (ld and col0 multiples of 8 elements).
template <typename Tin, int ROWS, int W, int LDS, int NT>
__device__ __forceinline__ void load_tile(float *dst, const Tin *src, long row0, int nc, int H,
                                          int h, int ld, int col0, int tid) {
    constexpr int VE = 16 / (int)sizeof(Tin);
    constexpr int VPR = W / VE;
    constexpr int NV = (ROWS * VPR + NT - 1) / NT;
    uint4 buf[NV];
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        const int e = tid + n * NT;
        const int t = e / VPR, vc = e % VPR;
        buf[n] = make_uint4(0u, 0u, 0u, 0u);
        if (e < ROWS * VPR && t < nc)
            buf[n] = *reinterpret_cast<const uint4 *>(
                src + ((size_t)(row0 + t) * H + h) * ld + col0 + vc * VE);
    }
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        const int e = tid + n * NT;
        if (e < ROWS * VPR) {
            const int t = e / VPR, vc = e % VPR;
            float f[VE];
            unpack16(buf[n], f);
#pragma unroll
            for (int i = 0; i < VE; ++i) dst[t * LDS + vc * VE + i] = f[i];
        }
    }
}

// A dense fp32 block [ROWS][W] (row stride lds_src floats in global memory)
// into shared memory with row stride LDS; float4 loads, all issued first.
template <int ROWS, int W, int LDS, int NT>
__device__ __forceinline__ void load_block_f32(float *dst, const float *src, int lds_src,
                                               int tid) {
    constexpr int VPR = W / 4;
    constexpr int NV = (ROWS * VPR + NT - 1) / NT;
    float4 buf[NV];
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        const int e = tid + n * NT;
        buf[n] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < ROWS * VPR)
            buf[n] = *reinterpret_cast<const float4 *>(src + (size_t)(e / VPR) * lds_src +
                                                       (e % VPR) * 4);
    }
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        const int e = tid + n * NT;
        if (e < ROWS * VPR) {
            float *d = dst + (e / VPR) * LDS + (e % VPR) * 4;
            d[0] = buf[n].x; d[1] = buf[n].y; d[2] = buf[n].z; d[3] = buf[n].w;
        }
    }
}

}  // namespace kla
