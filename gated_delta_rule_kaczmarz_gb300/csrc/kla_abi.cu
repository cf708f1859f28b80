// C ABI of the library (declared in include/kla.h): host-side validation,
// path selection and launches.  No device memory is allocated here.

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "../../include/kla.h"
#include "kla_internal.h"

namespace kla {
static std::atomic<unsigned long long> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
}  // namespace kla

namespace {

thread_local std::string g_last_error;

kla_status fail(kla_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

kla_status ok() {
    g_last_error.clear();
    return KLA_OK;
}

kla_status cuda_fail(cudaError_t e, const char *what) {
    return fail(KLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Host-side fault hook for tests: KLA_FAULT_INJECT=launch makes every
// launching entry point report KLA_ERR_CUDA before touching the device.
bool inject_launch_fault() {
    const char *s = std::getenv("KLA_FAULT_INJECT");
    return s != nullptr && std::strcmp(s, "launch") == 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Common size/dtype checks.  Returns KLA_OK or the failure status.
kla_status check_shape(int H, int dk, int dv, int chunk, int dtype) {
    if (H <= 0 || dk <= 0 || dv <= 0 || chunk <= 0)
        return fail(KLA_ERR_INVALID_ARG, "sizes must be positive (H=%d dk=%d dv=%d chunk=%d)",
                    H, dk, dv, chunk);
    if (dtype != KLA_DTYPE_F32 && dtype != KLA_DTYPE_BF16)
        return fail(KLA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (dk != dv || (dk != 64 && dk != 128))
        return fail(KLA_ERR_UNSUPPORTED, "supported head sizes: dk == dv in {64,128} (got %d,%d)",
                    dk, dv);
    if (chunk != kla::kChunk)
        return fail(KLA_ERR_UNSUPPORTED, "supported chunk length: 64 (got %d)", chunk);
    return KLA_OK;
}

// The tensor-core path needs at least one full 64-row TMA box of tokens.
bool use_tc_path(int d, int dtype, long total_T) {
    return total_T >= kla::kChunk && kla::chunk_tc_supported(d, dtype);
}

long chunks_upper(long n_seq, long total_T) {
    // every sequence adds at most one partial chunk
    return (total_T + kla::kChunk - 1) / kla::kChunk + n_seq;
}

// Number of chunk slots a call needs: exact for fixed length, an upper bound
// for varlen.
long n_chunks(bool varlen, long n_seq, long T, long total_T) {
    return varlen ? chunks_upper(n_seq, total_T) : n_seq * ((T + kla::kChunk - 1) / kla::kChunk);
}

size_t ws_bytes(bool varlen, long n_seq, long T, long total_T, int H, int d, int dtype) {
    if (use_tc_path(d, dtype, total_T))
        return kla::kWsHeader +
               kla::chunk_tc_workspace_bytes(n_chunks(varlen, n_seq, T, total_T), H, (int)n_seq) +
               (varlen ? 0 : kla::chunk_tc_split_bytes((int)n_seq, (int)T, H));
    return varlen ? kla::kWsHeader : 0;
}

// Writes S_T for calls with no tokens: S_T = S0 (or zeros).
kla_status states_only(const float *S0, float *S_T, size_t n, cudaStream_t s) {
    if (!S_T || n == 0) return ok();
    cudaError_t e = S0 ? (S0 == S_T ? cudaSuccess
                                    : cudaMemcpyAsync(S_T, S0, n * sizeof(float),
                                                      cudaMemcpyDeviceToDevice, s))
                       : cudaMemsetAsync(S_T, 0, n * sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(e, "state copy");
    return ok();
}

kla_status run_prefill(kla::Problem &p, bool varlen, void *workspace, size_t workspace_bytes,
                       cudaStream_t s) {
    const size_t need = ws_bytes(varlen, p.n_seq, p.T, p.total_T, p.H, p.d, p.dtype);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need)
            return fail(KLA_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                        workspace ? workspace_bytes : (size_t)0);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(KLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
        p.status = static_cast<unsigned *>(workspace);
        p.ws = static_cast<unsigned char *>(workspace) + kla::kWsHeader;
        p.ws_bytes = workspace_bytes - kla::kWsHeader;
    } else {
        // a path that needs no workspace still records its status in one the
        // caller passes, so that kla_workspace_status reads this call's
        p.status = (workspace != nullptr && workspace_bytes >= sizeof(unsigned) &&
                    (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0)
                       ? static_cast<unsigned *>(workspace)
                       : nullptr;
        p.ws = nullptr;
        p.ws_bytes = 0;
    }
    if (inject_launch_fault()) return fail(KLA_ERR_CUDA, "injected launch fault (KLA_FAULT_INJECT)");

    cudaError_t e = cudaSuccess;
    const bool tc = use_tc_path(p.d, p.dtype, p.total_T);
    if (p.status) {
        // varlen: a device check of cu_seqlens writes the status (the
        // tensor-core path does it in its own preparation kernel)
        if (varlen && !tc) {
            e = kla::launch_check_seqlens(p, s);
        } else {
            const size_t reset =
                tc ? kla::chunk_tc_reset_bytes(p, n_chunks(varlen, p.n_seq, p.T, p.total_T)) : 0;
            e = cudaMemsetAsync(p.status, 0, reset ? kla::kWsHeader + reset : sizeof(unsigned), s);
        }
        if (e != cudaSuccess) return cuda_fail(e, "status init");
    }
    if (tc) {
        e = kla::launch_chunk_tc(p, n_chunks(varlen, p.n_seq, p.T, p.total_T), s);
    } else {
        e = kla::launch_chunk_simt(p, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return ok();
}

}  // namespace

namespace kla {
void set_error_message(const char *msg) { g_last_error = msg; }
}  // namespace kla

namespace {
// Shared by the fixed-length and varlen backward entries (cu_seqlens NULL:
// fixed length, n_seq = B, T given).
int run_bwd(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
            float eps, const float *S0, const void *d_o, const float *dS_T, void *dq, void *dk,
            void *dv, float *dalpha, float *deta, float *dS0, const int *cu_seqlens, int n_seq,
            int T, int total_T, int H, int dk_, int dv_, int chunk, int dtype, int beta_mode,
            void *workspace, size_t workspace_bytes, void *stream) {
    kla_status st = check_shape(H, dk_, dv_, chunk, dtype);
    if (st != KLA_OK) return st;
    if (beta_mode != KLA_BETA_KACZMARZ && beta_mode != KLA_BETA_GIVEN)
        return fail(KLA_ERR_INVALID_ARG, "unknown beta_mode %d", beta_mode);
    if (!(eps >= 0.f)) return fail(KLA_ERR_INVALID_ARG, "eps must be >= 0");
    const long rows = total_T;
    if ((long)n_seq * H > INT32_MAX)
        return fail(KLA_ERR_UNSUPPORTED, "problem too large (sequences x H must fit in int32)");
    if (dalpha && !alpha)
        return fail(KLA_ERR_INVALID_ARG, "dalpha requires alpha (no decay has no alpha gradient)");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(d_o) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv) || !aligned4(alpha) || !aligned4(eta) ||
        !aligned4(dalpha) || !aligned4(deta) || !aligned16(S0) || !aligned16(dS_T) ||
        !aligned16(dS0))
        return fail(KLA_ERR_INVALID_ARG,
                    "q, k, v, d_o, dq, dk, dv and the states must be 16-byte aligned, the "
                    "per-token gates 4-byte");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows == 0 || n_seq == 0) {   // no tokens: dS0 = dS_T
        if (inject_launch_fault()) return fail(KLA_ERR_CUDA, "injected launch fault (KLA_FAULT_INJECT)");
        return states_only(dS_T, dS0, (size_t)n_seq * H * dk_ * dv_, s);
    }
    if (!q || !k || !v || !eta || !d_o || !dq || !dk || !dv)
        return fail(KLA_ERR_INVALID_ARG, "q, k, v, eta, d_o, dq, dk and dv must be non-null");
    const size_t need = kla::kWsHeader + kla::chunk_bwd_workspace_bytes(
                                             cu_seqlens != nullptr, n_seq, T, total_T, H, dk_,
                                             dtype);
    if (workspace == nullptr || workspace_bytes < need)
        return fail(KLA_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(KLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (inject_launch_fault()) return fail(KLA_ERR_CUDA, "injected launch fault (KLA_FAULT_INJECT)");
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(unsigned), s);   // status word
    if (e != cudaSuccess) return cuda_fail(e, "status init");
    kla::BwdProblem p{};
    p.q = q; p.k = k; p.v = v; p.dout = d_o; p.alpha = alpha; p.eta = eta; p.S0 = S0;
    p.dS_T = dS_T; p.eps = eps; p.dq = dq; p.dk = dk; p.dv = dv; p.dalpha = dalpha;
    p.deta = deta; p.dS0 = dS0; p.n_seq = n_seq; p.T = T; p.total_T = total_T;
    p.cu_seqlens = cu_seqlens; p.H = H; p.d = dk_; p.dtype = dtype;
    p.beta_mode = beta_mode;
    p.status = static_cast<unsigned *>(workspace);
    p.ws = static_cast<unsigned char *>(workspace) + kla::kWsHeader;
    e = kla::launch_chunk_bwd(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return ok();
}
}  // namespace

extern "C" {

const char *kla_status_str(int status) {
    switch (status) {
        case KLA_OK: return "ok";
        case KLA_ERR_INVALID_ARG: return "invalid argument";
        case KLA_ERR_UNSUPPORTED: return "unsupported size or dtype";
        case KLA_ERR_CUDA: return "CUDA error";
        case KLA_ERR_TIMEOUT: return "device wait timed out";
        case KLA_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

const char *kla_last_error_message(void) { return g_last_error.c_str(); }

int kla_version(void) { return 100; }

unsigned long long kla_launch_count(void) { return kla::g_launches.load(std::memory_order_relaxed); }

size_t kla_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk, int dtype) {
    if (B < 0 || T < 0) return 0;
    if (check_shape(H, dk, dv, chunk, dtype) != KLA_OK) return 0;
    return ws_bytes(false, B, T, (long)B * T, H, dk, dtype);
}

size_t kla_chunk_fwd_varlen_workspace_size(int N, int total_T, int H, int dk, int dv, int chunk,
                                           int dtype) {
    if (N < 0 || total_T < 0) return 0;
    if (check_shape(H, dk, dv, chunk, dtype) != KLA_OK) return 0;
    return ws_bytes(true, N, 0, total_T, H, dk, dtype);
}

int kla_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *alpha,
                     const float *eta, float eps, const float *S0, void *o, float *S_T, int B,
                     int T, int H, int dk, int dv, int chunk, int dtype, int beta_mode,
                     void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || T < 0) return fail(KLA_ERR_INVALID_ARG, "negative size (B=%d T=%d)", B, T);
    kla_status st = check_shape(H, dk, dv, chunk, dtype);
    if (st != KLA_OK) return st;
    if (beta_mode != KLA_BETA_KACZMARZ && beta_mode != KLA_BETA_GIVEN)
        return fail(KLA_ERR_INVALID_ARG, "unknown beta_mode %d", beta_mode);
    if (!(eps >= 0.f)) return fail(KLA_ERR_INVALID_ARG, "eps must be >= 0");
    const long rows = (long)B * T;
    if (rows > INT32_MAX || (long)B * H > INT32_MAX)
        return fail(KLA_ERR_UNSUPPORTED, "problem too large (B*T and B*H must fit in int32)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t nstate = (size_t)B * H * dk * dv;
    if ((S0 && !aligned16(S0)) || (S_T && !aligned16(S_T)))
        return fail(KLA_ERR_INVALID_ARG, "state pointers must be 16-byte aligned");
    if (rows == 0) {
        if (inject_launch_fault()) return fail(KLA_ERR_CUDA, "injected launch fault (KLA_FAULT_INJECT)");
        return states_only(S0, S_T, nstate, s);
    }
    if (!q || !k || !v || !eta || !o)
        return fail(KLA_ERR_INVALID_ARG, "q, k, v, eta and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(alpha) ||
        !aligned4(eta))
        return fail(KLA_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned, alpha and eta 4-byte");
    kla::Problem p{};
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.eta = eta; p.eps = eps;
    p.S0 = S0; p.o = o; p.S_T = S_T; p.cu_seqlens = nullptr;
    p.n_seq = B; p.T = T; p.total_T = (int)rows; p.H = H; p.d = dk; p.dtype = dtype;
    p.beta_mode = beta_mode;
    return run_prefill(p, false, workspace, workspace_bytes, s);
}

int kla_chunk_fwd(const void *q, const void *k, const void *v, const float *alpha,
                  const float *eta, float eps, const float *S0, void *o, float *S_T, int B,
                  int T, int H, int dk, int dv, int chunk, int dtype, void *workspace,
                  size_t workspace_bytes, void *stream) {
    return kla_chunk_fwd_ex(q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, dk, dv, chunk, dtype,
                            KLA_BETA_KACZMARZ, workspace, workspace_bytes, stream);
}

int kla_chunk_fwd_varlen_ex(const void *q, const void *k, const void *v, const float *alpha,
                            const float *eta, float eps, const float *S0, void *o, float *S_T,
                            const int *cu_seqlens, int N, int total_T, int H, int dk, int dv,
                            int chunk, int dtype, int beta_mode, void *workspace,
                            size_t workspace_bytes, void *stream) {
    if (N < 0 || total_T < 0)
        return fail(KLA_ERR_INVALID_ARG, "negative size (N=%d total_T=%d)", N, total_T);
    kla_status st = check_shape(H, dk, dv, chunk, dtype);
    if (st != KLA_OK) return st;
    if (beta_mode != KLA_BETA_KACZMARZ && beta_mode != KLA_BETA_GIVEN)
        return fail(KLA_ERR_INVALID_ARG, "unknown beta_mode %d", beta_mode);
    if (!(eps >= 0.f)) return fail(KLA_ERR_INVALID_ARG, "eps must be >= 0");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((S0 && !aligned16(S0)) || (S_T && !aligned16(S_T)))
        return fail(KLA_ERR_INVALID_ARG, "state pointers must be 16-byte aligned");
    if (N == 0) {
        if (total_T != 0) return fail(KLA_ERR_INVALID_ARG, "N == 0 requires total_T == 0");
        return ok();
    }
    if (!cu_seqlens) return fail(KLA_ERR_INVALID_ARG, "cu_seqlens must be non-null");
    if (total_T > 0) {
        if (!q || !k || !v || !eta || !o)
            return fail(KLA_ERR_INVALID_ARG, "q, k, v, eta and o must be non-null");
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
            !aligned4(alpha) || !aligned4(eta))
            return fail(KLA_ERR_INVALID_ARG,
                        "q, k, v, o must be 16-byte aligned, alpha and eta 4-byte");
    }
    kla::Problem p{};
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.eta = eta; p.eps = eps;
    p.S0 = S0; p.o = o; p.S_T = S_T; p.cu_seqlens = cu_seqlens;
    p.n_seq = N; p.T = 0; p.total_T = total_T; p.H = H; p.d = dk; p.dtype = dtype;
    p.beta_mode = beta_mode;
    return run_prefill(p, true, workspace, workspace_bytes, s);
}

int kla_chunk_fwd_varlen(const void *q, const void *k, const void *v, const float *alpha,
                         const float *eta, float eps, const float *S0, void *o, float *S_T,
                         const int *cu_seqlens, int N, int total_T, int H, int dk, int dv,
                         int chunk, int dtype, void *workspace, size_t workspace_bytes,
                         void *stream) {
    return kla_chunk_fwd_varlen_ex(q, k, v, alpha, eta, eps, S0, o, S_T, cu_seqlens, N, total_T,
                                   H, dk, dv, chunk, dtype, KLA_BETA_KACZMARZ, workspace,
                                   workspace_bytes, stream);
}

int kla_decode_step_ex(const void *q, const void *k, const void *v, const float *alpha,
                       const float *eta, float eps, float *S, void *o, int B, int H, int dk,
                       int dv, int dtype, int beta_mode, void *stream) {
    if (B < 0) return fail(KLA_ERR_INVALID_ARG, "negative batch");
    kla_status st = check_shape(H, dk, dv, kla::kChunk, dtype);
    if (st != KLA_OK) return st;
    if (beta_mode != KLA_BETA_KACZMARZ && beta_mode != KLA_BETA_GIVEN)
        return fail(KLA_ERR_INVALID_ARG, "unknown beta_mode %d", beta_mode);
    if (!(eps >= 0.f)) return fail(KLA_ERR_INVALID_ARG, "eps must be >= 0");
    if (B == 0) return ok();
    if (!q || !k || !v || !eta || !S || !o)
        return fail(KLA_ERR_INVALID_ARG, "q, k, v, eta, S and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(S) || !aligned16(o) ||
        !aligned4(alpha) || !aligned4(eta))
        return fail(KLA_ERR_INVALID_ARG,
                    "q, k, v, S, o must be 16-byte aligned, alpha and eta 4-byte");
    if ((long)B * H > INT32_MAX) return fail(KLA_ERR_UNSUPPORTED, "B*H too large");
    if (inject_launch_fault()) return fail(KLA_ERR_CUDA, "injected launch fault (KLA_FAULT_INJECT)");
    cudaError_t e = kla::launch_decode(q, k, v, alpha, eta, eps, S, o, B * H, dk, dtype,
                                       beta_mode, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ok();
}

int kla_decode_step(const void *q, const void *k, const void *v, const float *alpha,
                    const float *eta, float eps, float *S, void *o, int B, int H, int dk, int dv,
                    int dtype, void *stream) {
    return kla_decode_step_ex(q, k, v, alpha, eta, eps, S, o, B, H, dk, dv, dtype,
                              KLA_BETA_KACZMARZ, stream);
}

size_t kla_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dtype) {
    if (B < 0 || T < 0) return 0;
    if (check_shape(H, dk, dk, kla::kChunk, dtype) != KLA_OK) return 0;
    return kla::kWsHeader +
           kla::chunk_bwd_workspace_bytes(false, B, T, (int)((long)B * T), H, dk, dtype);
}

size_t kla_chunk_bwd_varlen_workspace_size(int N, int total_T, int H, int dk, int dtype) {
    if (N < 0 || total_T < 0) return 0;
    if (check_shape(H, dk, dk, kla::kChunk, dtype) != KLA_OK) return 0;
    return kla::kWsHeader + kla::chunk_bwd_workspace_bytes(true, N, 0, total_T, H, dk, dtype);
}

int kla_chunk_bwd(const void *q, const void *k, const void *v, const float *alpha,
                  const float *eta, float eps, const float *S0, const void *d_o,
                  const float *dS_T, void *dq, void *dk, void *dv, float *dalpha, float *deta,
                  float *dS0, int B, int T, int H, int dk_, int dv_, int chunk, int dtype,
                  int beta_mode, void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || T < 0) return fail(KLA_ERR_INVALID_ARG, "negative size (B=%d T=%d)", B, T);
    if ((long)B * T > INT32_MAX)
        return fail(KLA_ERR_UNSUPPORTED, "problem too large (B*T must fit in int32)");
    return run_bwd(q, k, v, alpha, eta, eps, S0, d_o, dS_T, dq, dk, dv, dalpha, deta, dS0,
                   nullptr, B, T, (int)((long)B * T), H, dk_, dv_, chunk, dtype, beta_mode,
                   workspace, workspace_bytes, stream);
}

int kla_chunk_bwd_varlen(const void *q, const void *k, const void *v, const float *alpha,
                         const float *eta, float eps, const float *S0, const void *d_o,
                         const float *dS_T, void *dq, void *dk, void *dv, float *dalpha,
                         float *deta, float *dS0, const int *cu_seqlens, int N, int total_T,
                         int H, int dk_, int dv_, int chunk, int dtype, int beta_mode,
                         void *workspace, size_t workspace_bytes, void *stream) {
    if (N < 0 || total_T < 0)
        return fail(KLA_ERR_INVALID_ARG, "negative size (N=%d total_T=%d)", N, total_T);
    if (N > 0 && total_T > 0 && !cu_seqlens)
        return fail(KLA_ERR_INVALID_ARG, "cu_seqlens must be non-null");
    if (!aligned4(cu_seqlens)) return fail(KLA_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
    return run_bwd(q, k, v, alpha, eta, eps, S0, d_o, dS_T, dq, dk, dv, dalpha, deta, dS0,
                   cu_seqlens, N, 0, total_T, H, dk_, dv_, chunk, dtype, beta_mode, workspace,
                   workspace_bytes, stream);
}

size_t kla_ccq_query_workspace_size(int B, int T, int H, int dk, int dtype) {
    if (B < 0 || T < 0) return 0;
    if (check_shape(H, dk, dk, kla::kChunk, dtype) != KLA_OK) return 0;
    return kla::ccq_workspace_bytes(B, T, H, dk, dtype);
}

int kla_ccq_query(const void *q, const void *k, const float *lambda, const float *Ms0,
                  const float *ms0, const float *ns0, void *q_clean, float *Ms_T, float *ms_T,
                  float *ns_T, int B, int T, int H, int dk, int dtype, void *workspace,
                  size_t workspace_bytes, void *stream) {
    if (B < 0 || T < 0) return fail(KLA_ERR_INVALID_ARG, "negative size (B=%d T=%d)", B, T);
    kla_status st = check_shape(H, dk, dk, kla::kChunk, dtype);
    if (st != KLA_OK) return st;
    if ((long)B * T > INT32_MAX || (long)B * H > INT32_MAX)
        return fail(KLA_ERR_UNSUPPORTED, "problem too large (B*T and B*H must fit in int32)");
    if ((long)B * T > 0 && (!q || !k || !lambda || !q_clean))
        return fail(KLA_ERR_INVALID_ARG, "q, k, lambda and q_clean must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(q_clean) || !aligned4(lambda) ||
        !aligned4(Ms0) || !aligned4(ms0) || !aligned4(ns0) || !aligned4(Ms_T) ||
        !aligned4(ms_T) || !aligned4(ns_T))
        return fail(KLA_ERR_INVALID_ARG, "q, k, q_clean must be 16-byte aligned, the rest 4-byte");
    const size_t need = kla::ccq_workspace_bytes(B, T, H, dk, dtype);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need))
        return fail(KLA_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(KLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (inject_launch_fault()) return fail(KLA_ERR_CUDA, "injected launch fault (KLA_FAULT_INJECT)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if ((long)B * T == 0) {
        // no tokens: the statistics pass through
        const size_t nM = (size_t)B * H * dk * dk, nm = (size_t)B * H * dk, nn = (size_t)B * H;
        if (Ms_T && e == cudaSuccess)
            e = Ms0 ? cudaMemcpyAsync(Ms_T, Ms0, nM * 4, cudaMemcpyDeviceToDevice, s)
                    : cudaMemsetAsync(Ms_T, 0, nM * 4, s);
        if (ms_T && e == cudaSuccess)
            e = ms0 ? cudaMemcpyAsync(ms_T, ms0, nm * 4, cudaMemcpyDeviceToDevice, s)
                    : cudaMemsetAsync(ms_T, 0, nm * 4, s);
        if (ns_T && e == cudaSuccess)
            e = ns0 ? cudaMemcpyAsync(ns_T, ns0, nn * 4, cudaMemcpyDeviceToDevice, s)
                    : cudaMemsetAsync(ns_T, 0, nn * 4, s);
        if (e != cudaSuccess) return cuda_fail(e, "statistics copy");
        return ok();
    }
    kla::CcqProblem p{};
    p.q = q; p.k = k; p.lambda = lambda; p.Ms0 = Ms0; p.ms0 = ms0; p.ns0 = ns0;
    p.q_clean = q_clean; p.Ms_T = Ms_T; p.ms_T = ms_T; p.ns_T = ns_T;
    p.B = B; p.T = T; p.H = H; p.d = dk; p.dtype = dtype; p.ws = workspace;
    e = kla::launch_ccq(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "ccq launch");
    return ok();
}

int kla_ccq_query_step(const void *q, const void *k, const float *lambda, float *Ms, float *ms,
                       float *ns, void *q_clean, int B, int H, int dk, int dtype, void *stream) {
    if (B < 0) return fail(KLA_ERR_INVALID_ARG, "negative batch");
    kla_status st = check_shape(H, dk, dk, kla::kChunk, dtype);
    if (st != KLA_OK) return st;
    if (B == 0) return ok();
    if (!q || !k || !lambda || !Ms || !ms || !ns || !q_clean)
        return fail(KLA_ERR_INVALID_ARG, "all pointers must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(q_clean) || !aligned4(lambda) ||
        !aligned4(Ms) || !aligned4(ms) || !aligned4(ns))
        return fail(KLA_ERR_INVALID_ARG, "q, k, q_clean must be 16-byte aligned, the rest 4-byte");
    if ((long)B * H > INT32_MAX) return fail(KLA_ERR_UNSUPPORTED, "B*H too large");
    if (inject_launch_fault()) return fail(KLA_ERR_CUDA, "injected launch fault (KLA_FAULT_INJECT)");
    cudaError_t e = kla::launch_ccq_step(q, k, lambda, Ms, ms, ns, q_clean, B * H, dk, dtype,
                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ccq step launch");
    return ok();
}

int kla_workspace_status(const void *workspace, size_t workspace_bytes, void *stream) {
    if (workspace == nullptr || workspace_bytes < kla::kWsHeader) return ok();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned word = 0;
    e = cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (word == kla::kDevOk) return ok();
    if (word == kla::kDevBadSeqlens)
        return fail(KLA_ERR_INVALID_ARG, "cu_seqlens rejected on the device");
    if (word == kla::kDevTimeout) return fail(KLA_ERR_TIMEOUT, "a device-side wait timed out");
    return fail(KLA_ERR_CUDA, "unknown device status %u", word);
}

}  // extern "C"
