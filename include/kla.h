/*
 * kla.h -- C ABI of the GB300 (sm_103a) Kaczmarz Linear Attention library.
 *
 * The operation (Kaczmarz Linear Attention summary, gist.science
 * 2605.08587, section "A Regra de Atualizacao KLA"), per (sequence, head),
 * for t = 1..T, with a state S in R^{dk x dv} (section "Implementacao"):
 *
 *     beta_t = eta_t / (||k_t||^2 + eps)          (0 when the sum is 0)
 *     S~     = alpha_t S_{t-1}                    (Gated DeltaNet scalar decay)
 *     e_t    = v_t - S~^T k_t
 *     S_t    = S~ + beta_t k_t e_t^T
 *     o_t    = S_t^T q_t                          (read after the write)
 *
 * kla_chunk_fwd / kla_chunk_fwd_varlen compute it with the chunkwise-parallel
 * (blockwise) algorithm that the summary says KLA keeps from Gated DeltaNet,
 * with B = Diag(beta_1..beta_C) in the block solver (section
 * "Implementacao"); kla_decode_step applies one token to stored states (the
 * recurrent form behind the decode throughput of section "Eficiencia").
 *
 * Conventions for every entry point
 *   - Tensors are dense, row-major, in device memory, owned by the caller.
 *     The library never allocates, frees or retains device memory and keeps
 *     no pointer after a call returns.
 *   - `dtype` (kla_dtype) is the storage type of q, k, v and o.  alpha, eta
 *     and the states are always fp32.  Arithmetic is fp32 (bf16 tensor-core
 *     products with fp32 accumulation on the bf16 prefill path).
 *   - Supported: dk == dv in {64, 128}, chunk == 64.  Other sizes return
 *     KLA_ERR_UNSUPPORTED without launching anything.
 *   - alpha must lie in (0, 1] and eps >= 0 (values are not scanned; outside
 *     that range results are unspecified but every access stays in bounds).
 *     alpha may be NULL: alpha_t = 1 for every token (no decay, DeltaNet's
 *     recurrence).
 *   - The *_ex entry points take a write-coefficient mode (kla_beta_mode):
 *     KLA_BETA_KACZMARZ is the rule above; KLA_BETA_GIVEN uses beta_t = eta_t
 *     itself, the learned write strength of Gated DeltaNet that KLA replaces
 *     (KLA summary, "Contribuicoes Principais" item 2 and "Implementacao":
 *     only B = Diag(beta) of the block solver changes).  With alpha == NULL
 *     and KLA_BETA_GIVEN the calls compute DeltaNet.  The entry points
 *     without _ex use KLA_BETA_KACZMARZ.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: a KLA_OK return means the work was validated and
 *     enqueued; faults of the enqueued work surface on a later
 *     synchronisation, and device-detected argument errors through
 *     kla_workspace_status().
 *   - Errors are returned as kla_status codes; nothing is thrown or aborted
 *     across the ABI.  kla_last_error_message() gives a one-line detail for
 *     the calling thread's last failure.
 *   - q, k, v, o and the states must be 16-byte aligned, alpha and eta 4-byte
 *     aligned; o and S_T may not alias inputs
 *     except that S_T may equal S0.
 */
#ifndef KLA_H
#define KLA_H

#include <stddef.h>

#if defined(__GNUC__)
#define KLA_API __attribute__((visibility("default")))
#else
#define KLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KLA_OK = 0,
    KLA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, negative size, bad cu_seqlens */
    KLA_ERR_UNSUPPORTED = 2,   /* valid request outside the supported set */
    KLA_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute, ...) */
    KLA_ERR_TIMEOUT = 4,       /* a bounded device-side wait gave up */
    KLA_ERR_WORKSPACE = 5      /* workspace missing or smaller than required */
} kla_status;

typedef enum {
    KLA_DTYPE_F32 = 0,
    KLA_DTYPE_BF16 = 1
} kla_dtype;

typedef enum {
    KLA_BETA_KACZMARZ = 0,     /* beta_t = eta_t / (||k_t||^2 + eps), 0 if the sum is 0 */
    KLA_BETA_GIVEN = 1         /* beta_t = eta_t */
} kla_beta_mode;

/* Static string for a status code; never NULL. */
KLA_API const char *kla_status_str(int status);

/* One-line description of the calling thread's most recent failure
 * ("" if none).  Valid until the next call on the same thread. */
KLA_API const char *kla_last_error_message(void);

/* Library version, major*10000 + minor*100 + patch. */
KLA_API int kla_version(void);

/* Number of CUDA kernels this library has enqueued since it was loaded
 * (all threads, all devices).  Lets a caller count device work per call. */
KLA_API unsigned long long kla_launch_count(void);

/*
 * Workspace bytes that kla_chunk_fwd needs for these sizes (0 when the
 * chosen path needs none, in which case `workspace` may be NULL).  Returns 0
 * as well for unsupported sizes; the call then reports the reason.
 */
KLA_API size_t kla_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv,
                                    int chunk, int dtype);

/*
 * Chunkwise prefill over a fixed-length batch.
 *   q, k     : [B, T, H, dk]  dtype
 *   v        : [B, T, H, dv]  dtype
 *   alpha    : [B, T, H]      fp32 decay, in (0, 1]
 *   eta      : [B, T, H]      fp32 relaxation gate
 *   eps      : scalar stabiliser added once to ||k_t||^2
 *   S0       : [B, H, dk, dv] fp32 initial states (dv fastest) or NULL = 0
 *   o        : [B, T, H, dv]  dtype, written
 *   S_T      : [B, H, dk, dv] fp32 final states, written; NULL = not needed;
 *              may equal S0 (in-place state update)
 *   workspace: device buffer of at least kla_chunk_fwd_workspace_size(...)
 *              bytes, 256-byte aligned, owned by the caller; contents on
 *              entry are ignored.  One workspace must not be shared by calls
 *              that may run concurrently.
 * T == 0 or B == 0 is valid and writes only S_T (= S0, or zeros).
 *
 * Execution (bf16, dk = dv = 128, B*T >= 64): the tensor-core kernels, as one
 * cooperative launch when the state pass of every (batch, head) fits on half
 * of the SMs and each sequence has an even number of chunks, else as two.
 * Few heads with long sequences (T a multiple of 128) run the sequence split:
 * each sequence as P <= 8 segments of whole 128-token tiles, as equal as the
 * tile count allows (at least 1024 tokens each, or 4096 with one CTA per
 * chain), P chosen for the shortest chain among those whose state and
 * transition passes fit on the SMs at once; the segments' start states are
 * chained and their outputs corrected (four launches, or three when fused,
 * which needs equal segments).  The environment variable KLA_SEQ_SPLIT=P
 * forces a factor up to T / 128 (1 disables the split); the workspace size depends on that
 * choice and on the SM count of the current device, so query it on the device
 * and with the environment of the call.  In two launches, the state pass runs
 * one CTA per (sequence, head) instead of two when two per head would
 * outnumber the SMs (KLA_WIDE_STATE=0 or 1 forces either; results agree to
 * rounding).  Other dtypes and sizes run on the CUDA cores (fp32 arithmetic).
 */
KLA_API int kla_chunk_fwd(const void *q, const void *k, const void *v,
                  const float *alpha, const float *eta, float eps,
                  const float *S0, void *o, float *S_T,
                  int B, int T, int H, int dk, int dv, int chunk, int dtype,
                  void *workspace, size_t workspace_bytes, void *stream);

/* kla_chunk_fwd with a write-coefficient mode (kla_beta_mode); an unknown
 * mode returns KLA_ERR_INVALID_ARG.  Same workspace size. */
KLA_API int kla_chunk_fwd_ex(const void *q, const void *k, const void *v,
                             const float *alpha, const float *eta, float eps,
                             const float *S0, void *o, float *S_T,
                             int B, int T, int H, int dk, int dv, int chunk, int dtype,
                             int beta_mode, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Workspace bytes for kla_chunk_fwd_varlen (see kla_chunk_fwd_workspace_size). */
KLA_API size_t kla_chunk_fwd_varlen_workspace_size(int N, int total_T, int H, int dk,
                                           int dv, int chunk, int dtype);

/*
 * Chunkwise prefill over N packed sequences of different lengths.
 *   q, k       : [total_T, H, dk]   v, o : [total_T, H, dv]
 *   alpha, eta : [total_T, H]
 *   cu_seqlens : device int32 [N + 1]; sequence n is token rows
 *                cu_seqlens[n] .. cu_seqlens[n+1]-1.  Must satisfy
 *                cu_seqlens[0] == 0, non-decreasing, cu_seqlens[N] == total_T.
 *                The device checks this; a violation skips all work and is
 *                reported by kla_workspace_status() as KLA_ERR_INVALID_ARG.
 *                Empty sequences are allowed (their S_T is S0, or zeros).
 *   S0, S_T    : [N, H, dk, dv] fp32 (S0 NULL = zero, S_T NULL = not needed)
 * Chunks never straddle sequence boundaries; every sequence's last chunk
 * may be partial.
 */
KLA_API int kla_chunk_fwd_varlen(const void *q, const void *k, const void *v,
                         const float *alpha, const float *eta, float eps,
                         const float *S0, void *o, float *S_T,
                         const int *cu_seqlens, int N, int total_T,
                         int H, int dk, int dv, int chunk, int dtype,
                         void *workspace, size_t workspace_bytes, void *stream);

/* kla_chunk_fwd_varlen with a write-coefficient mode (kla_beta_mode). */
KLA_API int kla_chunk_fwd_varlen_ex(const void *q, const void *k, const void *v,
                                    const float *alpha, const float *eta, float eps,
                                    const float *S0, void *o, float *S_T,
                                    const int *cu_seqlens, int N, int total_T,
                                    int H, int dk, int dv, int chunk, int dtype,
                                    int beta_mode, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * One decode step: one new token for each of B*H (sequence, head) states,
 * updated in place.
 *   q, k       : [B, H, dk]  dtype     v, o : [B, H, dv] dtype
 *   alpha, eta : [B, H] fp32
 *   S          : [B, H, dk, dv] fp32, read and overwritten with S_t
 * Each state is read once and written once.
 */
KLA_API int kla_decode_step(const void *q, const void *k, const void *v,
                    const float *alpha, const float *eta, float eps,
                    float *S, void *o, int B, int H, int dk, int dv, int dtype,
                    void *stream);

/* kla_decode_step with a write-coefficient mode (kla_beta_mode). */
KLA_API int kla_decode_step_ex(const void *q, const void *k, const void *v,
                               const float *alpha, const float *eta, float eps,
                               float *S, void *o, int B, int H, int dk, int dv,
                               int dtype, int beta_mode, void *stream);

/*
 * Size in bytes of the device array that kla_chunk_fwd_noalloc uses as its
 * workspace (64 MiB).  Every GPU that loads this library holds it until the
 * process exits.
 */
#define KLA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * kla_chunk_fwd without a workspace argument: the same computation, results
 * and errors as kla_chunk_fwd, for callers that cannot allocate device memory
 * when they run the prefill (a framework that owns all device memory through
 * its own pool, a plugin interface that is handed only input and output
 * pointers, or a serving loop that cannot afford cudaMalloc's device-wide
 * synchronisation).  The pages this library follows have no counterpart of
 * this call; it is a deployment convenience.
 *   - It allocates nothing.  Its scratch is one file-scope device array of
 *     KLA_NOALLOC_SCRATCH_BYTES; sizes whose kla_chunk_fwd_workspace_size()
 *     exceeds that are rejected with KLA_ERR_WORKSPACE before any device work.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address and caches it; make that first call before any
 *     stream capture.
 *   - All calls share the array, which keeps the last call's contents (the
 *     status word it needs zeroed is cleared by every call).  Calls that
 *     overlap on the GPU race on it: serialise them on one stream.
 * Arguments are those of kla_chunk_fwd minus workspace and workspace_bytes.
 */
KLA_API int kla_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                  const float *alpha, const float *eta, float eps,
                                  const float *S0, void *o, float *S_T,
                                  int B, int T, int H, int dk, int dv, int chunk,
                                  int dtype, void *stream);

/*
 * Synchronises `stream` and returns the device status that the last
 * kla_chunk_fwd_noalloc call on the current device recorded in its built-in
 * array: KLA_OK or KLA_ERR_TIMEOUT (a bounded device-side wait gave up and
 * the outputs of that call are incomplete).  The counterpart of
 * kla_workspace_status for the call without a workspace; like that call it
 * has no counterpart in the pages.  KLA_ERR_CUDA if the array's address
 * cannot be looked up.
 */
KLA_API int kla_chunk_fwd_noalloc_status(void *stream);

/*
 * Backward pass of the fixed-length chunkwise forward (kla_chunk_fwd_ex with
 * the same inputs and beta_mode): the gradients of the scalar
 *
 *     L = sum_t <d_o_t, o_t> + <dS_T, S_T>
 *
 * with respect to every input, by reverse-mode differentiation of the
 * recurrence of the KLA summary (gist.science 2605.08587, "A Regra de
 * Atualizacao KLA"), including the path through beta_t's key norm
 * (d beta / d k = -2 eta k / (||k||^2 + eps)^2).  The chunk form it uses is
 * the derivative of the blockwise solver of the same summary's
 * "Implementacao" section.
 *   q, k, v, alpha, eta, eps, S0, beta_mode : as kla_chunk_fwd_ex
 *   d_o   : [B, T, H, dv] dtype, the gradient of o
 *   dS_T  : [B, H, dk, dv] fp32, the gradient of S_T, or NULL (zero)
 *   dq, dk, dv : [B, T, H, *] dtype (written)
 *   dalpha, deta : [B, T, H] fp32 (written unless NULL; dalpha must be NULL
 *           when alpha is NULL)
 *   dS0   : [B, H, dk, dv] fp32 (written unless NULL)
 *   workspace : kla_chunk_bwd_workspace_size(...) bytes, 256-byte aligned,
 *           owned by the caller; it starts with the device status word and
 *           holds the state and its gradient at every chunk boundary.
 * dk == dv in {64, 128}, chunk 64, fp32 or bf16; arithmetic fp32 on the CUDA
 * cores (three launches: the forward recording the chunk-start states, the
 * chain of state gradients over the chunks in reverse, the per-chunk token
 * gradients).  Asynchronous on `stream`.
 */
KLA_API size_t kla_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dtype);

/* Backward of kla_chunk_fwd_varlen_ex: packed q, k, v, d_o, dq, dk, dv
 * [total_T, H, *], alpha, eta, dalpha, deta [total_T, H], cu_seqlens int32
 * device [N + 1] (validated on the device: a bad table is reported by
 * kla_workspace_status as KLA_ERR_INVALID_ARG and no gradient is written),
 * S0, dS_T, dS0 [N, H, dk, dv]; otherwise as kla_chunk_bwd. */
KLA_API size_t kla_chunk_bwd_varlen_workspace_size(int N, int total_T, int H, int dk, int dtype);
KLA_API int kla_chunk_bwd_varlen(const void *q, const void *k, const void *v, const float *alpha,
                                 const float *eta, float eps, const float *S0, const void *d_o,
                                 const float *dS_T, void *dq, void *dk, void *dv, float *dalpha,
                                 float *deta, float *dS0, const int *cu_seqlens, int N,
                                 int total_T, int H, int dk_, int dv_, int chunk, int dtype,
                                 int beta_mode, void *workspace, size_t workspace_bytes,
                                 void *stream);
KLA_API int kla_chunk_bwd(const void *q, const void *k, const void *v, const float *alpha,
                          const float *eta, float eps, const float *S0, const void *d_o,
                          const float *dS_T, void *dq, void *dk, void *dv, float *dalpha,
                          float *deta, float *dS0, int B, int T, int H, int dk_, int dv_,
                          int chunk, int dtype, int beta_mode, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Curvature-Conditioned Query (CCQ) read-side contraction ("Don't Read
 * Everything: A Curvature-Conditioned Query for Linear Attention",
 * gist.science 2606.01294, sections "O Mecanismo" and "Integracao"):
 *
 *     Sigma_t   = M_t / n_t - mu_t mu_t^T,   mu_t = m_t / n_t
 *     q_clean_t = q_t - lambda_t Sigma_t q_t
 *
 * with the running statistics of the keys of each (sequence, head) up to and
 * including token t: M_t = sum k k^T (dk x dk), m_t = sum k (dk), n_t =
 * count.  The write rule is unchanged and the read is o_t = S_t^T q_clean_t,
 * so a CCQ layer is kla_chunk_fwd / kla_decode_step called with q_clean in
 * place of q.
 *   q, k, q_clean : [B, T, H, dk] dtype     lambda : [B, T, H] fp32 gate
 *   Ms0, Ms_T     : [B, H, dk, dk] fp32 (symmetric), ms0, ms_T : [B, H, dk],
 *   ns0, ns_T     : [B, H] fp32 counts; the initial statistics may be NULL
 *                   (zero), the final ones NULL (not needed).  Ms_T may not
 *                   alias Ms0 (likewise ms, ns).
 *   workspace     : kla_ccq_query_workspace_size(...) bytes, 256-byte
 *                   aligned, owned by the caller.  It starts with the device
 *                   status word (read with kla_workspace_status after the
 *                   call); the rest is scratch.
 * dk in {64, 128}.  bf16 inputs with dk = 128 (and B*T >= 64) take the tensor
 * cores: M_t q_t comes from the chunked forward's tcgen05 kernels run with
 * W = 0, U~ = K and no decay (products of bf16 values accumulated in fp32,
 * the carried M rounded to bf16 as the operand of its product with Q, M q
 * rounded to bf16 before the fp32 finish).  Other inputs: fp32 arithmetic
 * on the CUDA cores, the per-chunk M stored in the input dtype.
 */
KLA_API size_t kla_ccq_query_workspace_size(int B, int T, int H, int dk, int dtype);
KLA_API int kla_ccq_query(const void *q, const void *k, const float *lambda,
                          const float *Ms0, const float *ms0, const float *ns0,
                          void *q_clean, float *Ms_T, float *ms_T, float *ns_T,
                          int B, int T, int H, int dk, int dtype,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * One CCQ token per (b, h) for decoding: the statistics Ms [B, H, dk, dk],
 * ms [B, H, dk], ns [B, H] (fp32) are updated in place with k, then q_clean
 * [B, H, dk] = q - lambda Sigma q.  q, k: [B, H, dk]; lambda: [B, H].
 */
KLA_API int kla_ccq_query_step(const void *q, const void *k, const float *lambda, float *Ms,
                               float *ms, float *ns, void *q_clean, int B, int H, int dk,
                               int dtype, void *stream);

/*
 * Synchronises `stream` and returns the status that the last prefill call
 * using `workspace` recorded on the device: KLA_OK, KLA_ERR_INVALID_ARG
 * (cu_seqlens rejected) or KLA_ERR_TIMEOUT.  A workspace of 0 bytes (NULL)
 * has no status word and returns KLA_OK.  A prefill whose path needs no
 * workspace still records its status in a workspace the caller passes (at
 * least 4 bytes, 256-byte aligned).
 *
 * Every wait of one CTA on another (the single-launch prefill's state pass
 * waiting for a chunk pair to be published) and every wait on the CTA's own
 * asynchronous copies and tensor-core products is bounded (about one second
 * of SM clock).  A wait that runs out records KLA_ERR_TIMEOUT here; the CTA's
 * other warps stop waiting on work that will not come, the copies and
 * products it already issued are waited for (they complete by themselves),
 * its tensor memory is released and it leaves.  For tests only, the
 * environment variable KLA_TEST_FLAG_WAIT=<cycles> bounds the flag waits of
 * the single-launch prefill by that many cycles and makes its state pass
 * first wait on a header word that nothing sets, so that the wait runs out.
 */
KLA_API int kla_workspace_status(const void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KLA_H */
