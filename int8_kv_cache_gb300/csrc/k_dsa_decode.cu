// Instantiations of the decode kernel: DSA sparse-candidate decode.
#include "decode_launch.cuh"

namespace i8kv {
cudaError_t launch_dsa_decode(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                              KernelInfo* info) {
  return dispatch_decode<false, false, true>(key, p, s, info);
}
}  // namespace i8kv
