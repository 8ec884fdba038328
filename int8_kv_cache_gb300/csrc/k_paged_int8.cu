// Instantiations of the decode kernel: paged decode over an INT8 cache.
#include "decode_launch.cuh"

namespace i8kv {
cudaError_t launch_paged_int8(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                              KernelInfo* info) {
  return dispatch_decode<true, false, true>(key, p, s, info);
}
}  // namespace i8kv
