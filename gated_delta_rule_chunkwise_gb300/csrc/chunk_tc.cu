// Chunkwise forward on the tcgen05 tensor cores (bf16 operands, fp32 TMEM
// accumulators, fp32 state).  Not built yet: chunk_tc_supported() reports
// false, so LDN_VARIANT_AUTO routes every call to the fp32 SIMT kernel.
#include "ldn_internal.cuh"

namespace ldn {

bool chunk_tc_supported(const ChunkArgs &) { return false; }

cudaError_t launch_chunk_tc(const ChunkArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ldn
