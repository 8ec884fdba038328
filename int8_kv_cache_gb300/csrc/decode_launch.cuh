// Host-side launch of the decode kernel instantiations (one per translation
// unit includes this): the per-device shared-memory attributes, the
// occupancy / round query the geometry uses, and the launch with the
// programmatic-serialization attribute.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "decode_kernel.cuh"

namespace i8kv {

template <int D, int NT, bool PAGED, bool FP16C, bool PLO, bool FP8>
cudaError_t run_decode(const DecodeParams& p, cudaStream_t s, KernelInfo* info) {
  using T = Tile<D, NT, FP16C, PAGED || !PLO>;
  auto kern = decode_kernel<D, NT, PAGED, FP16C, PLO, FP8>;
  // the opt-in shared-memory size is a per-function attribute: set it once per device
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(done.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
    if (e != cudaSuccess) return e;
    // ask for the largest shared-memory carveout, so that the resident CTAs per
    // SM that the occupancy API reports are the ones the launch gets
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  if (info != nullptr) {
    info->round = T::kWarps * T::kStep;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&info->occupancy, kern, T::kThreads,
                                                         T::kSmem);
  }
  cudaLaunchConfig_t cfg = {};
  // (balanced pieces: ceil(num_splits / 2) CTAs per unit for num_splits slots)
  cfg.gridDim = dim3((unsigned)(p.rows * p.Hkv),
                     (unsigned)(p.balanced ? (p.num_splits + 1) / 2 : p.num_splits));
  cfg.blockDim = dim3(T::kThreads);
  cfg.dynamicSmemBytes = T::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool PAGED, bool FP16C, bool PLO, bool FP8 = false>
cudaError_t dispatch_decode(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                            KernelInfo* info) {
  switch (key.D * 10 + key.nt) {
    case 641: return run_decode<64, 1, PAGED, FP16C, PLO, FP8>(p, s, info);
    case 642: return run_decode<64, 2, PAGED, FP16C, PLO, FP8>(p, s, info);
    case 1281: return run_decode<128, 1, PAGED, FP16C, PLO, FP8>(p, s, info);
    case 1282: return run_decode<128, 2, PAGED, FP16C, PLO, FP8>(p, s, info);
    case 2561: return run_decode<256, 1, PAGED, FP16C, PLO, FP8>(p, s, info);
    case 2562: return run_decode<256, 2, PAGED, FP16C, PLO, FP8>(p, s, info);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace i8kv
