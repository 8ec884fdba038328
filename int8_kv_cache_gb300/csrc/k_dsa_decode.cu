// Instantiations of the decode kernels: DSA sparse-candidate decode (the mma.sync kernel, or the tensor-memory kernel when that engine is selected).
#include "decode_tc.cuh"

namespace i8kv {
cudaError_t launch_dsa_decode(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                           int* occupancy) {
  return key.tc ? dispatch_decode_tc<false, false>(key, p, s, occupancy)
                : dispatch_decode<false, false, true>(key, p, s, occupancy);
}
}  // namespace i8kv
