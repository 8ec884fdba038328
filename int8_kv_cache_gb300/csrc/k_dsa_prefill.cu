// Instantiations of the decode kernel: DSA sparse-candidate prefill (single fp16 probability tile).
#include "decode_launch.cuh"

namespace i8kv {
cudaError_t launch_dsa_prefill(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                           KernelInfo* info) {
  return dispatch_decode<false, false, false>(key, p, s, info);
}
}  // namespace i8kv
