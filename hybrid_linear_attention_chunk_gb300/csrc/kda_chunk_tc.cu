// Tensor-core chunked prefill (tcgen05 / TMEM / TMA) - not built yet.
#include "kda_internal.cuh"

namespace kda {

bool chunk_tc_supports(const PrefillArgs &) { return false; }

cudaError_t launch_chunk_tc(const PrefillArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kda
