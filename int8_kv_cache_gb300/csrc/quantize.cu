// Quantize-on-write: new key / value rows (fp16) into a paged INT8 cache
// (onnxruntime PR 29912, CUDA kernels: "ReshapeAndCache quantizes on write").
//   code[d] = clamp(round_half_even(x[d] / scale[g, d]), -127, 127)
// with the quotient computed by an IEEE fp32 division; a NaN quotient stores 0;
// slots outside [0, num_slots) write nothing (-1 is padding; other
// out-of-range slots raise I8KV_FLAG_BAD_SLOT).
// One thread per 8 channels of one (token, KV head) row: a 16-byte load of
// the fp16 row piece, the scales, an 8-byte store of the codes, for K and V.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/int8kv.h"
#include "device.cuh"
#include "internal.h"

namespace i8kv {

// codes of 8 fp16 values with 8 scales, packed into two 32-bit words
__device__ __forceinline__ uint2 quantize8(uint4 raw, const float (&s)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 f2 = __half22float2(h[j / 2]);
    const float x = (j & 1) ? f2.y : f2.x;
    float q = rintf(__fdiv_rn(x, s[j]));
    if (q != q) q = 0.f;  // NaN
    q = fminf(fmaxf(q, -127.f), 127.f);
    const uint32_t b = static_cast<uint32_t>(static_cast<int32_t>(q)) & 0xFFu;
    w[j / 4] |= b << (8 * (j % 4));
  }
  return make_uint2(w[0], w[1]);
}

__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const __half* __restrict__ kn, const __half* __restrict__ vn,
                         const int32_t* __restrict__ slots, long long rows, int Hkv, int D,
                         int8_t* __restrict__ kc, int8_t* __restrict__ vc, long long num_slots,
                         const float* __restrict__ ks, const float* __restrict__ vs,
                         int per_channel, uint32_t* flags) {
  grid_dependency_wait();
  const int cpr = D / 8;  // 8-channel pieces per row
  const long long pieces = rows * cpr;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < pieces;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / cpr;  // token * Hkv + g
    const int c = (int)(i - row * cpr);
    const long long n = row / Hkv;
    const int g = (int)(row - n * Hkv);
    const int slot = slots[n];
    if (slot < 0) continue;
    if ((long long)slot >= num_slots) {
      if (flags != nullptr && c == 0) atomicOr(flags, I8KV_FLAG_BAD_SLOT);
      continue;
    }
    const uint4 xk = *reinterpret_cast<const uint4*>(kn + row * D + c * 8);
    const uint4 xv = *reinterpret_cast<const uint4*>(vn + row * D + c * 8);
    float sk[8], sv[8];
    if (per_channel) {
      const float4* pk = reinterpret_cast<const float4*>(ks + (long long)g * D + c * 8);
      const float4* pv = reinterpret_cast<const float4*>(vs + (long long)g * D + c * 8);
      const float4 k0 = pk[0], k1 = pk[1], v0 = pv[0], v1 = pv[1];
      sk[0] = k0.x; sk[1] = k0.y; sk[2] = k0.z; sk[3] = k0.w;
      sk[4] = k1.x; sk[5] = k1.y; sk[6] = k1.z; sk[7] = k1.w;
      sv[0] = v0.x; sv[1] = v0.y; sv[2] = v0.z; sv[3] = v0.w;
      sv[4] = v1.x; sv[5] = v1.y; sv[6] = v1.z; sv[7] = v1.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        sk[j] = ks[0];
        sv[j] = vs[0];
      }
    }
    const long long dst = ((long long)slot * Hkv + g) * D + c * 8;
    *reinterpret_cast<uint2*>(kc + dst) = quantize8(xk, sk);
    *reinterpret_cast<uint2*>(vc + dst) = quantize8(xv, sv);
  }
}

cudaError_t launch_reshape_and_cache(const void* k_new, const void* v_new, const int32_t* slots,
                                     int num_tokens, int Hkv, int D, int8_t* k_cache,
                                     int8_t* v_cache, long long num_slots, const float* ks,
                                     const float* vs, int per_channel, uint32_t* flags,
                                     cudaStream_t stream) {
  const long long rows = (long long)num_tokens * Hkv;
  const long long pieces = rows * (D / 8);
  if (pieces == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long want = (pieces + 255) / 256;
  const long long cap = (long long)sms * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(want < cap ? want : cap));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel, reinterpret_cast<const __half*>(k_new),
                            reinterpret_cast<const __half*>(v_new), slots, rows, Hkv, D, k_cache,
                            v_cache, num_slots, ks, vs, per_channel, flags);
}

}  // namespace i8kv
