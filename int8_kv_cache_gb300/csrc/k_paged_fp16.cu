// Instantiations of the decode kernel: paged decode over an FP16 cache.
#include "decode_launch.cuh"

namespace i8kv {
cudaError_t launch_paged_fp16(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                           KernelInfo* info) {
  return dispatch_decode<true, true, true>(key, p, s, info);
}
}  // namespace i8kv
