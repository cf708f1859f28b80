// Tensor-core (tcgen05) chunkwise prefill: bf16 inputs, d = 128.
#include "kla_internal.h"

namespace kla {

bool chunk_tc_supported(int, int) { return false; }
size_t chunk_tc_workspace_bytes(long, int) { return 0; }
cudaError_t launch_chunk_tc(const Problem &, long, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kla
