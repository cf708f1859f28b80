// Single-token decode step on stored fp32 states.
//
// Kaczmarz Linear Attention summary (gist.science 2605.08587), section
// "A Regra de Atualizacao KLA", applied to one token on the state kept from
// earlier tokens (the recurrent form, O(1) per token, section "Eficiencia"):
//
//   y = S^T k,  z = S^T q                  (one read of S)
//   e = v - alpha y                        (residual against alpha S)
//   S <- alpha S + beta k e^T              (one write of S)
//   o = S_new^T q = alpha z + beta (k.q) e
//   beta = eta / (||k||^2 + eps), 0 when the denominator is 0 (or beta = eta
//   in the given-beta mode); alpha == NULL means alpha = 1
//
// The kernel is bound by HBM: each (b,h) state (dk*dv*4 bytes) is streamed in
// once and out once.  One CTA of 256 threads owns one state; every thread
// keeps its slice of S in registers between the reduction and the write, so
// the state is never re-read.  Thread tid holds the float4 column group
// tid % (d/4) of rows tid/(d/4) + i*(256/(d/4)).

#include <cuda_bf16.h>

#include "kla_internal.h"

namespace kla {
namespace {

__device__ __forceinline__ float ld_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_out(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

constexpr int kDecThreads = 256;

template <typename Tin, int D>
__global__ void __launch_bounds__(kDecThreads, 2)
decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
              const Tin *__restrict__ v, const float *__restrict__ alpha,
              const float *__restrict__ eta, float eps, int beta_given,
              float *__restrict__ S, Tin *__restrict__ o) {
    constexpr int C4 = D / 4;                 // float4 groups per state row
    constexpr int RSTEP = kDecThreads / C4;   // row stride between a thread's rows
    constexpr int R = D / RSTEP;              // rows per thread
    static_assert(R * RSTEP == D && RSTEP * C4 == kDecThreads, "tiling");

    __shared__ float ks[D], qs[D], es[D];
    __shared__ __align__(16) float red_y[RSTEP][D];
    __shared__ __align__(16) float red_z[RSTEP][D];
    __shared__ float scal[2];

    const int unit = blockIdx.x;
    const int tid = threadIdx.x;
    const int c4 = tid % C4;
    const int r0 = tid / C4;

    float4 *Sp = reinterpret_cast<float4 *>(S + (size_t)unit * D * D);

    // Issue every state load first: R independent 16-byte streaming loads.
    float4 s[R];
#pragma unroll
    for (int i = 0; i < R; ++i) s[i] = __ldcs(Sp + (size_t)(r0 + i * RSTEP) * C4 + c4);

    const size_t vbase = (size_t)unit * D;
    if (tid < D) {
        ks[tid] = ld_in(k, vbase + tid);
        qs[tid] = ld_in(q, vbase + tid);
    }
    const float a = alpha ? alpha[unit] : 1.f;   // no alpha: no decay
    const float et = eta[unit];
    __syncthreads();

    if (tid < 32) {  // ||k||^2 and k.q
        float n2 = 0.f, kq = 0.f;
#pragma unroll
        for (int i = tid; i < D; i += 32) {
            n2 = fmaf(ks[i], ks[i], n2);
            kq = fmaf(ks[i], qs[i], kq);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            n2 += __shfl_xor_sync(0xffffffffu, n2, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }
        if (tid == 0) {
            const float den = n2 + eps;
            scal[0] = beta_given ? et : ((den == 0.f) ? 0.f : et / den);
            scal[1] = kq;
        }
    }

    float4 y = make_float4(0.f, 0.f, 0.f, 0.f), z = y;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const float kr = ks[r0 + i * RSTEP], qr = qs[r0 + i * RSTEP];
        y.x = fmaf(s[i].x, kr, y.x); y.y = fmaf(s[i].y, kr, y.y);
        y.z = fmaf(s[i].z, kr, y.z); y.w = fmaf(s[i].w, kr, y.w);
        z.x = fmaf(s[i].x, qr, z.x); z.y = fmaf(s[i].y, qr, z.y);
        z.z = fmaf(s[i].z, qr, z.z); z.w = fmaf(s[i].w, qr, z.w);
    }
    reinterpret_cast<float4 *>(&red_y[r0][0])[c4] = y;
    reinterpret_cast<float4 *>(&red_z[r0][0])[c4] = z;
    __syncthreads();

    const float beta = scal[0];
    if (tid < D) {
        float yy = 0.f, zz = 0.f;
#pragma unroll
        for (int g = 0; g < RSTEP; ++g) {
            yy += red_y[g][tid];
            zz += red_z[g][tid];
        }
        const float e = ld_in(v, vbase + tid) - a * yy;
        es[tid] = e;
        st_out(o, vbase + tid, fmaf(beta * scal[1], e, a * zz));
    }
    __syncthreads();

    const float4 e4 = reinterpret_cast<const float4 *>(es)[c4];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const float bk = beta * ks[r0 + i * RSTEP];
        float4 w;
        w.x = fmaf(bk, e4.x, a * s[i].x);
        w.y = fmaf(bk, e4.y, a * s[i].y);
        w.z = fmaf(bk, e4.z, a * s[i].z);
        w.w = fmaf(bk, e4.w, a * s[i].w);
        __stcs(Sp + (size_t)(r0 + i * RSTEP) * C4 + c4, w);
    }
}

template <typename Tin, int D>
cudaError_t launch_t(const void *q, const void *k, const void *v, const float *alpha,
                     const float *eta, float eps, int beta_mode, float *S, void *o, int BH,
                     cudaStream_t s) {
    decode_kernel<Tin, D><<<BH, kDecThreads, 0, s>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k),
        static_cast<const Tin *>(v), alpha, eta, eps, beta_mode, S, static_cast<Tin *>(o));
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *alpha, const float *eta, float eps,
                          float *S, void *o, int BH, int d, int dtype, int beta_mode,
                          cudaStream_t s) {
    if (BH == 0) return cudaSuccess;
    if (dtype == 1) {
        if (d == 128) return launch_t<__nv_bfloat16, 128>(q, k, v, alpha, eta, eps, beta_mode, S, o, BH, s);
        return launch_t<__nv_bfloat16, 64>(q, k, v, alpha, eta, eps, beta_mode, S, o, BH, s);
    }
    if (d == 128) return launch_t<float, 128>(q, k, v, alpha, eta, eps, beta_mode, S, o, BH, s);
    return launch_t<float, 64>(q, k, v, alpha, eta, eps, beta_mode, S, o, BH, s);
}

}  // namespace kla
