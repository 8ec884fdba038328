// dsa_decode_static_workspace: the sparse-candidate decode for callers that
// cannot allocate device memory when they call us.
//
// Some callers have no way to obtain a scratch buffer at call time: an
// inference engine's per-step "enqueue" hook that must not allocate (an
// allocation there can block on the device, or is simply forbidden by the
// host framework), code without access to the application's memory allocator,
// or latency-critical loops that must never touch the allocator.  For them the
// split workspace lives in a fixed device array that is part of this library
// (below).  It is allocated once, when CUDA loads the library's device code on
// a device, and stays allocated on every device that loaded it until the
// process exits.
//
// Everything else is the ordinary dsa_decode: this entry point only supplies
// the scratch pointer.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/int8kv.h"

namespace {

// The scratch: split partials of at most I8KV_STATIC_WORKSPACE_BYTES bytes.
static __device__ __align__(256) unsigned char g_static_workspace[I8KV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device.  The symbol's name in
// host code is not a device address, so it is resolved with
// cudaGetSymbolAddress once per device, with that device current, and cached.
// The cache assumes the device's primary context lives as long as the process
// (no cudaDeviceReset in between): a reset unloads the array with the module.
i8kv_status static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return I8KV_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return I8KV_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr) return I8KV_ECUDA;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return I8KV_OK;
}

}  // namespace

extern "C" i8kv_status dsa_decode_static_workspace(
    const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache, const float* k_scale,
    const float* v_scale, int32_t scale_kind, const int32_t* idx, int32_t S, int32_t Hq,
    int32_t Hkv, int32_t D, int64_t N, int32_t max_sel, float softmax_scale,
    const float* head_sink, int32_t num_splits, int32_t chunk, uint16_t* out, float* lse,
    uint32_t* flags, void* stream) {
  // Nothing in the scratch has to start at zero: the decode kernel writes the
  // (m, l) entry of every (unit, split, head) that the combine reads, and the
  // combine reads a split's accumulator only when that split wrote it.  So no
  // clearing is needed between calls, and the previous call's contents are
  // never read.
  // With out == NULL dsa_decode would leave the partials in the array below,
  // where the caller cannot read them: refuse it.
  if (out == nullptr && S > 0) return I8KV_EINVAL;
  void* ws = nullptr;
  i8kv_status st = static_workspace(&ws);
  if (st != I8KV_OK) return st;
  // dsa_decode checks the geometry's workspace need against the fixed size and
  // returns I8KV_EWORKSPACE, before enqueuing anything, when it does not fit.
  return dsa_decode(q, k_cache, v_cache, k_scale, v_scale, scale_kind, idx, S, Hq, Hkv, D, N,
                    max_sel, softmax_scale, head_sink, num_splits, chunk, ws,
                    I8KV_STATIC_WORKSPACE_BYTES, out, lse, flags, stream);
}
