// Log-sum-exp combine of split partials with the head sink, and the
// stand-alone int8 -> fp16 conversion kernel.
//
// Combine (onnxruntime PR 33707, Summary of Changes §2: the merge of the
// split-K partials; onnxruntime PR 29912, CUDA kernels: ApplyHeadSink):
//   M = max_k m_k;  L = sum_k l_k e^(m_k - M);  O = sum_k acc_k e^(m_k - M) / L;
//   lse = M + ln L;  O <- O / (1 + e^(s_h - lse)).
// One warp per (unit, query head): lane k holds split k's (m, l) (at most 32
// splits), the warp reduces M and L with shuffles, then every lane accumulates
// D/32 channels over the splits with vector loads.  Splits with m = -inf are
// skipped without reading their accumulator.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"

namespace i8kv {

template <int D>
__global__ void __launch_bounds__(128)
combine_kernel(const float* __restrict__ acc, const float* __restrict__ m,
               const float* __restrict__ l, int units, int ns, int Hkv, int G,
               const float* __restrict__ sink, __half* __restrict__ out, float* __restrict__ lse) {
  constexpr int V = D / 32;  // channels per lane: 2, 4 or 8
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= units * G) return;
  const int u = wid / G, j = wid - (wid / G) * G;
  const long long ml0 = (long long)u * ns * G + j;  // split k at ml0 + k*G

  const float mk = lane < ns ? m[ml0 + (long long)lane * G] : neg_inf();
  const float lk = lane < ns ? l[ml0 + (long long)lane * G] : 0.f;
  float M = mk;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float f = (mk == neg_inf()) ? 0.f : fast_exp2((mk - M) * kLog2e);
  float L = f * lk;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);

  float o[V];
#pragma unroll
  for (int i = 0; i < V; ++i) o[i] = 0.f;
  for (int k = 0; k < ns; ++k) {
    const float fk = __shfl_sync(0xffffffffu, f, k);
    if (fk == 0.f) continue;  // warp-uniform
    const float* src = acc + (((long long)u * ns + k) * G + j) * D + lane * V;
    if constexpr (V == 2) {
      const float2 a = *reinterpret_cast<const float2*>(src);
      o[0] += fk * a.x; o[1] += fk * a.y;
    } else {
#pragma unroll
      for (int i = 0; i < V; i += 4) {
        const float4 a = *reinterpret_cast<const float4*>(src + i);
        o[i] += fk * a.x; o[i + 1] += fk * a.y; o[i + 2] += fk * a.z; o[i + 3] += fk * a.w;
      }
    }
  }
  const int h = (u % Hkv) * G + j;
  float lse_v = neg_inf(), scale = 0.f;
  if (L > 0.f) {
    lse_v = M + logf(L);
    scale = 1.f / L;
    if (sink != nullptr) scale *= 1.f / (1.f + expf(sink[h] - lse_v));
  }
  __half* dst = out + (long long)wid * D + lane * V;
#pragma unroll
  for (int i = 0; i < V; i += 2) {
    *reinterpret_cast<__half2*>(dst + i) = __floats2half2_rn(o[i] * scale, o[i + 1] * scale);
  }
  if (lane == 0 && lse != nullptr) lse[wid] = lse_v;
}

cudaError_t launch_combine(const float* acc, const float* m, const float* l, int units,
                           int num_splits, int Hq, int Hkv, int D, const float* sink, void* out,
                           float* lse, cudaStream_t stream) {
  const int G = Hq / Hkv;
  const long long warps = (long long)units * G;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((warps + 3) / 4);
  __half* o = reinterpret_cast<__half*>(out);
  switch (D) {
    case 64: combine_kernel<64><<<blocks, 128, 0, stream>>>(acc, m, l, units, num_splits, Hkv, G, sink, o, lse); break;
    case 128: combine_kernel<128><<<blocks, 128, 0, stream>>>(acc, m, l, units, num_splits, Hkv, G, sink, o, lse); break;
    case 256: combine_kernel<256><<<blocks, 128, 0, stream>>>(acc, m, l, units, num_splits, Hkv, G, sink, o, lse); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Each thread converts four codes with the decode kernels' conversion.
__global__ void int8_to_fp16_kernel(const uint32_t* __restrict__ in, uint2* __restrict__ out,
                                    long long nwords) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nwords;
       i += (long long)gridDim.x * blockDim.x) {
    const uint32_t x = flip_i8x4(in[i]);
    out[i] = make_uint2(i8x2_to_h2(x, 0x4140u), i8x2_to_h2(x, 0x4342u));
  }
}

cudaError_t launch_int8_to_fp16(const int8_t* in, uint16_t* out, int64_t n, cudaStream_t stream) {
  const long long nwords = n / 4;
  if (nwords == 0) return cudaSuccess;
  const long long want = (nwords + 255) / 256;
  const unsigned blocks = (unsigned)(want < 4096 ? want : 4096);
  int8_to_fp16_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(in),
                                                   reinterpret_cast<uint2*>(out), nwords);
  return cudaGetLastError();
}

}  // namespace i8kv
