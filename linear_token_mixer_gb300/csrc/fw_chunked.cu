// fw_chunked.cu -- chunked tensor-core prefill (placeholder until the tcgen05
// kernel lands: it declines every call, so the recurrent kernel serves all).
#include "fw_internal.cuh"

namespace fw {
bool chunked_supported(const PrefillArgs &) { return false; }
cudaError_t launch_chunked(const PrefillArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fw
