// Instantiations of the decode kernels: paged decode over an INT8 cache (the mma.sync kernel, or the tensor-memory kernel when that engine is selected).
#include "decode_tc.cuh"

namespace i8kv {
cudaError_t launch_paged_int8(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                           int* occupancy) {
  return key.tc ? dispatch_decode_tc<true, false>(key, p, s, occupancy)
                : dispatch_decode<true, false, true>(key, p, s, occupancy);
}
}  // namespace i8kv
