// Log-sum-exp combine of split partials with the head sink, and the
// stand-alone int8 -> fp16 conversion kernel.
//
// Combine (onnxruntime PR 33707, Summary of Changes §2: the merge of the
// split-K partials; onnxruntime PR 29912, CUDA kernels: ApplyHeadSink):
//   M = max_k m_k;  L = sum_k l_k e^(m_k - M);  O = sum_k acc_k e^(m_k - M) / L;
//   lse = M + ln L;  O <- O / (1 + e^(s_h - lse)).
// One 128-thread CTA per (unit, query head): every thread owns D/128 channels
// (one or two; half the threads idle at D = 64) and issues the loads of all its
// splits at once, so the whole merge costs one L2 round trip.  Each warp reads
// the (m, l) of all splits (lane k holds split k) and reduces M and L with
// shuffles.  The accumulator of a split with m = -inf (an empty split, never
// written) is loaded with the others but selected away, never multiplied.
// The head's sink logit is loaded together with the partials.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"

namespace i8kv {

constexpr int kCombineThreads = 128;

template <int D>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const float* __restrict__ acc, const float* __restrict__ m,
               const float* __restrict__ l, int units, int ns, int Hkv, int G,
               const float* __restrict__ sink, __half* __restrict__ out, float* __restrict__ lse) {
  constexpr int V = D >= kCombineThreads ? D / kCombineThreads : 1;  // channels per thread
  const int wid = blockIdx.x;  // (unit, head) pair
  const int lane = threadIdx.x & 31;
  grid_dependency_wait();  // the partials come from the preceding decode kernel
  const int u = wid / G, j = wid - (wid / G) * G;
  const long long ml0 = (long long)u * ns * G + j;  // split k at ml0 + k*G
  const int c0 = threadIdx.x * V;                    // first channel of this thread
  const bool has = c0 < D;
  const int h = (u % Hkv) * G + j;                   // query head within the row
  // the sink logit travels with the partials' loads (one round trip in all)
  const float sink_h = sink != nullptr ? sink[h] : 0.f;

  // all loads first: (m, l) of every split, and this thread's accumulator
  // channels of every split (up to 32)
  const float mk = lane < ns ? m[ml0 + (long long)lane * G] : neg_inf();
  const float lk = lane < ns ? l[ml0 + (long long)lane * G] : 0.f;
  float a[32][V];
  const float* base = acc + ((long long)u * ns * G + j) * D + c0;
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    if (k < ns && has) {
      const float* src = base + (long long)k * G * D;
      if constexpr (V == 2) {
        const float2 v = *reinterpret_cast<const float2*>(src);
        a[k][0] = v.x;
        a[k][1] = v.y;
      } else {
        a[k][0] = *src;
      }
    }
  }
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
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    if (k < ns) {
      const float fk = __shfl_sync(0xffffffffu, f, k);
      // an empty split (fk = 0) may hold anything: select, do not multiply
#pragma unroll
      for (int i = 0; i < V; ++i) o[i] += fk != 0.f ? fk * a[k][i] : 0.f;
    }
  }
  if (!has) return;
  float lse_v = neg_inf(), scale = 0.f;
  if (L > 0.f) {
    lse_v = M + logf(L);
    scale = 1.f / L;
    if (sink != nullptr) scale *= 1.f / (1.f + expf(sink_h - lse_v));
  }
  __half* dst = out + (long long)wid * D + c0;
  if constexpr (V == 2) {
    *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(o[0] * scale, o[1] * scale);
  } else {
    *dst = __float2half_rn(o[0] * scale);
  }
  if (threadIdx.x == 0 && lse != nullptr) lse[wid] = lse_v;
}

cudaError_t launch_combine(const float* acc, const float* m, const float* l, int units,
                           int num_splits, int Hq, int Hkv, int D, const float* sink, void* out,
                           float* lse, cudaStream_t stream) {
  const int G = Hq / Hkv;
  const long long pairs = (long long)units * G;
  if (pairs == 0) return cudaSuccess;
  __half* o = reinterpret_cast<__half*>(out);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pairs);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (D) {
    case 64: return cudaLaunchKernelEx(&cfg, combine_kernel<64>, acc, m, l, units, num_splits, Hkv, G, sink, o, lse);
    case 128: return cudaLaunchKernelEx(&cfg, combine_kernel<128>, acc, m, l, units, num_splits, Hkv, G, sink, o, lse);
    case 256: return cudaLaunchKernelEx(&cfg, combine_kernel<256>, acc, m, l, units, num_splits, Hkv, G, sink, o, lse);
    default: return cudaErrorInvalidValue;
  }
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
