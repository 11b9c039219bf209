// bf16 tensor-core prefill (tcgen05): placeholder until the kernel lands.
#include "kda_internal.h"

namespace kda {
cudaError_t launch_chunk_fwd_bf16_tc(const ChunkArgs &, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace kda
