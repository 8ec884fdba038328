// Instantiations of the decode kernel: paged decode over an INT8 cache.
#include "decode_kernel.cuh"

namespace i8kv {
cudaError_t launch_paged_int8(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                              int* occupancy) {
  return dispatch_decode<true, false, true>(key, p, s, occupancy);
}
}  // namespace i8kv
