// Internal declarations shared by the ABI layer and the kernel files.
// Not part of the public interface (include/kla.h is).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace kla {

constexpr int kChunk = 64;             // chunk length C of the blockwise algorithm
constexpr size_t kWsHeader = 256;      // status word area at the start of a workspace

// Device status codes written into the workspace header (word 0).
enum DevStatus : unsigned {
    kDevOk = 0,
    kDevBadSeqlens = 1,
    kDevTimeout = 2,
};

// One prefill request after host validation.  Token row r of head h of a
// [*, H, d] tensor sits at (r * H + h) * d.  Sequence n (fixed length: batch
// index) covers rows seq_start(n) .. seq_start(n) + seq_len(n) - 1.
struct Problem {
    const void *q, *k, *v;
    const float *alpha, *eta;
    float eps;
    const float *S0;
    void *o;
    float *S_T;
    const int *cu_seqlens;   // device; nullptr for fixed length
    int n_seq;               // B (fixed) or N (varlen)
    int T;                   // fixed length (unused for varlen)
    int total_T;             // total token rows
    int H, d;                // heads, dk == dv
    int dtype;               // kla_dtype
    int beta_mode;           // 0: beta = eta / (||k||^2 + eps); 1: beta = eta
    void *S_chk;             // the state at every chunk start for the backward pass, or
                             // nullptr; slot = chunk * H + head.  CUDA-core path: [slots, d, d]
                             // fp32; tensor-core path: per slot the two 16 KB images of the
                             // bf16 128 x 64 operand tiles of the state's column halves
                             // (128-byte swizzle), as the state pass holds them
    const int *chunk_prefix; // CUDA-core varlen recording: first chunk of each sequence
    void *T_chk;             // tensor-core path with S_chk: T of every chunk slot
                             // ([slots, 64, 64] bf16), or nullptr
    unsigned *status;        // device status word, or nullptr
    void *ws;                // workspace after the header (path specific)
    size_t ws_bytes;
};

// Counts kernel launches made by the library (kla_launch_count()).
void note_launch(int n = 1);

// Sets the calling thread's kla_last_error_message() text.
void set_error_message(const char *msg);

// Kernel-file entry points; each returns cudaSuccess or the launch error.
cudaError_t launch_check_seqlens(const Problem &p, cudaStream_t s);
cudaError_t launch_chunk_simt(const Problem &p, cudaStream_t s);
cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *alpha, const float *eta, float eps,
                          float *S, void *o, int BH, int d, int dtype, int beta_mode,
                          cudaStream_t s);

// CCQ query contraction (kla_ccq.cu): q_clean for a fixed-length batch, and
// the one-token step with the statistics updated in place.
struct CcqProblem {
    const void *q, *k;
    const float *lambda;
    const float *Ms0, *ms0, *ns0;   // initial statistics or nullptr (zero)
    void *q_clean;
    float *Ms_T, *ms_T, *ns_T;      // final statistics or nullptr
    int B, T, H, d, dtype;
    void *ws;                       // ccq_workspace_bytes(B, T, H, d, dtype)
};
size_t ccq_workspace_bytes(int B, int T, int H, int d, int dtype);
cudaError_t launch_ccq(const CcqProblem &p, cudaStream_t s);
cudaError_t launch_ccq_step(const void *q, const void *k, const float *lambda, float *Ms,
                            float *ms, float *ns, void *q_clean, int BH, int d, int dtype,
                            cudaStream_t s);

// Backward of the chunkwise forward (kla_chunk_bwd.cu), fixed length or varlen.
struct BwdProblem {
    const void *q, *k, *v, *dout;
    const float *alpha, *eta, *S0, *dS_T;
    float eps;
    void *dq, *dk, *dv;
    float *dalpha, *deta, *dS0;
    int n_seq;               // B (fixed) or N (varlen)
    int T;                   // fixed length (unused for varlen)
    int total_T;             // token rows
    const int *cu_seqlens;   // device, varlen only
    int H, d, dtype, beta_mode;
    unsigned *status;
    void *ws;                // chunk_bwd_workspace_bytes(...) after the header
    // set by the launcher: the chunk tables (varlen)
    const int *chunk_prefix, *chunk_seq;
};
size_t chunk_bwd_workspace_bytes(bool varlen, int n_seq, int T, int total_T, int H, int d,
                                 int dtype);
cudaError_t launch_chunk_bwd(const BwdProblem &p, cudaStream_t s);

// Tensor-core (tcgen05) prefill for bf16, d = 128.
size_t chunk_tc_workspace_bytes(long n_chunks_upper, int H, int n_seq);
// The g [slots][64] fp32, W [slots][64][128] bf16 and A^T [slots][64][64] bf16
// arrays inside a tensor-core workspace (after its header).
void chunk_tc_ws_views(void *ws, long n_chunks_upper, int H, int n_seq, float **g, void **W,
                       void **A);
// Extra workspace bytes of a fixed-length batch that runs with the sequence
// split (0 when it does not).
size_t chunk_tc_split_bytes(int n_seq, int T, int H);
bool chunk_tc_supported(int d, int dtype);
cudaError_t launch_chunk_tc(const Problem &p, long n_chunks_upper, cudaStream_t s);
// Bytes after the workspace header that must be zero when launch_chunk_tc
// starts (the single-launch path's ready flags); cleared with the status word.
size_t chunk_tc_reset_bytes(const Problem &p, long n_chunks_upper);

}  // namespace kla
