// kda_chunk_tc.cu -- tensor-core chunked KDA forward (placeholder until the
// fused kernel lands: reports "not supported" so the dispatcher uses the
// token-recurrent kernel).
#include "kda_common.cuh"

namespace kda {
bool chunk_tc_supported(const FwdParams&, bool) { return false; }
cudaError_t launch_chunk_tc_fwd(const FwdParams&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kda
