// Instantiations of the decode kernel: paged decode over an FP16 cache.
#include "decode_kernel.cuh"

namespace i8kv {
cudaError_t launch_paged_fp16(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                           int* occupancy) {
  return dispatch_decode<true, true, true>(key, p, s, occupancy);
}
}  // namespace i8kv
