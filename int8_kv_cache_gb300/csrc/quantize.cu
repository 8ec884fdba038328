// Quantize-on-write: new key / value rows (fp16) into a paged INT8 or float8
// e4m3fn cache (onnxruntime PR 29912, CUDA kernels: "ReshapeAndCache quantizes
// on write"; Schema: cache element type int8 or float8e4m3fn).
//   INT8:   code[d] = clamp(round_half_even(x[d] / scale[g, d]), -127, 127)
//   e4m3fn: code[d] = the nearest e4m3fn value of x[d] / scale[g, d] (ties to
//           even), saturated to +-448
// where x / scale is the IEEE fp32 quotient; a NaN quotient stores 0; slots
// outside [0, num_slots) write nothing (-1 is padding; other out-of-range slots
// raise I8KV_FLAG_BAD_SLOT).
//
// The quotient is formed as x * r with r = 1/scale correctly rounded, which is
// within |q| * 2^-22 of the fp32 quotient fl(x / scale) (two roundings of 2^-24
// each, against one).  Rounding to a code is monotone, so when the codes of
// x*r*(1 - 2^-21) and x*r*(1 + 2^-21) agree they are also the code of
// fl(x / scale); only a quotient that close to a rounding boundary takes the
// division itself.
//
// Each thread owns one 8-channel piece (KV head g, channels 8c .. 8c+7) and
// walks the tokens two at a time, so that it forms the reciprocals of the
// piece's scales once: 16-byte loads of the fp16 row pieces (issued before the
// slots they go to are known) and 8-byte stores of the codes, for K and V.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/int8kv.h"
#include "device.cuh"
#include "internal.h"

namespace i8kv {

namespace {

constexpr float kLoBound = 1.f - 0x1p-21f;
constexpr float kHiBound = 1.f + 0x1p-21f;

__device__ __forceinline__ float int8_code(float q) {
  return fminf(fmaxf(rintf(q), -127.f), 127.f);
}

// Two floats -> two float8 e4m3fn bytes (lo in bits 0..7), nearest even,
// saturating to the largest finite magnitude.
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float nan_to_zero(float q) { return q != q ? 0.f : q; }

__device__ __forceinline__ uint32_t int8_byte(float c) {
  return static_cast<uint32_t>(static_cast<int32_t>(c)) & 0xFFu;
}

// Codes of 8 fp16 values (channel j in byte j % 4 of word j / 4) from the
// fp32 quotients x[j] / s[j * s_step] themselves: the exact path, taken for a
// piece with a quotient near a rounding boundary.
template <bool FP8>
__device__ __noinline__ uint2 quantize8_exact(uint4 raw, const float* __restrict__ s,
                                              int s_step) {
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float2 x = __half22float2(h[j / 2]);
    const float q0 = nan_to_zero(__fdiv_rn(x.x, s[j * s_step]));
    const float q1 = nan_to_zero(__fdiv_rn(x.y, s[(j + 1) * s_step]));
    const uint32_t b = FP8 ? e4m3x2_of(q0, q1) : int8_byte(int8_code(q0)) | (int8_byte(int8_code(q1)) << 8);
    w[j / 4] |= b << (8 * (j % 4));
  }
  return make_uint2(w[0], w[1]);
}

// The same codes from x[j] * r[j], r the correctly rounded reciprocals; a piece
// where some product lies within its error bound of a rounding boundary goes
// to the exact path.  INT8: the boundaries are the half-integers, so the test
// is | |q - rint(q)| - 1/2 | <= |q| 2^-21.  e4m3fn: the codes of q (1 -+ 2^-21)
// must agree.
template <bool FP8>
__device__ __forceinline__ uint2 quantize8(uint4 raw, const float* __restrict__ s, int s_step,
                                           const float (&r)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
  uint32_t w[2] = {0u, 0u};
  bool near = false;
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float2 x = __half22float2(h[j / 2]);
    const float q0 = nan_to_zero(x.x * r[j]), q1 = nan_to_zero(x.y * r[j + 1]);
    uint32_t b;
    if constexpr (FP8) {
      b = e4m3x2_of(q0 * kLoBound, q1 * kLoBound);
      near |= b != e4m3x2_of(q0 * kHiBound, q1 * kHiBound);
    } else {
      const float n0 = rintf(q0), n1 = rintf(q1);
      near |= fabsf(fabsf(q0 - n0) - 0.5f) <= fabsf(q0) * 0x1p-21f;
      near |= fabsf(fabsf(q1 - n1) - 0.5f) <= fabsf(q1) * 0x1p-21f;
      b = int8_byte(fminf(fmaxf(n0, -127.f), 127.f)) |
          (int8_byte(fminf(fmaxf(n1, -127.f), 127.f)) << 8);
    }
    w[j / 4] |= b << (8 * (j % 4));
  }
  if (near) return quantize8_exact<FP8>(raw, s, s_step);
  return make_uint2(w[0], w[1]);
}

constexpr int kQuantThreads = 256;
constexpr int kQuantBlocksPerSm = 4;

template <bool FP8>
__global__ void __launch_bounds__(kQuantThreads, kQuantBlocksPerSm)
reshape_and_cache_kernel(const __half* __restrict__ kn, const __half* __restrict__ vn,
                         const int32_t* __restrict__ slots, int num_tokens, int Hkv, int D,
                         uint8_t* __restrict__ kc, uint8_t* __restrict__ vc, long long num_slots,
                         const float* __restrict__ ks, const float* __restrict__ vs,
                         int per_channel, long long lanes, uint32_t* flags) {
  grid_dependency_wait();
  const int cpr = D / 8;                       // 8-channel pieces per (token, head) row
  const long long ppt = (long long)Hkv * cpr;  // pieces per token
  const long long row = ppt * 8;               // elements per token
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (tid >= lanes * ppt) return;
  const int piece = (int)(tid % ppt);          // fixed for this thread
  const int g = piece / cpr, c = piece - (piece / cpr) * cpr;
  const long long off = (long long)g * D + c * 8;
  const float* sk = per_channel ? ks + off : ks;
  const float* sv = per_channel ? vs + off : vs;
  const int step = per_channel ? 1 : 0;
  float rk[8], rv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    rk[j] = __frcp_rn(sk[j * step]);
    rv[j] = __frcp_rn(sv[j * step]);
  }
  auto store = [&](int slot, uint4 xk, uint4 xv) {
    if (slot < 0) return;
    if ((long long)slot >= num_slots) {
      if (flags != nullptr && piece == 0) atomicOr(flags, I8KV_FLAG_BAD_SLOT);
      return;
    }
    const long long dst = (long long)slot * row + off;
    *reinterpret_cast<uint2*>(kc + dst) = quantize8<FP8>(xk, sk, step, rk);
    *reinterpret_cast<uint2*>(vc + dst) = quantize8<FP8>(xv, sv, step, rv);
  };
  // two tokens per pass, their rows and slots all loaded before any use
  for (long long n = tid / ppt; n < num_tokens; n += 2 * lanes) {
    const long long n2 = n + lanes;
    const bool two = n2 < num_tokens;
    const uint4 xk0 = *reinterpret_cast<const uint4*>(kn + n * row + off);
    const uint4 xv0 = *reinterpret_cast<const uint4*>(vn + n * row + off);
    uint4 xk1 = make_uint4(0u, 0u, 0u, 0u), xv1 = xk1;
    if (two) {
      xk1 = *reinterpret_cast<const uint4*>(kn + n2 * row + off);
      xv1 = *reinterpret_cast<const uint4*>(vn + n2 * row + off);
    }
    const int s0 = slots[n];
    const int s1 = two ? slots[n2] : -1;
    store(s0, xk0, xv0);
    store(s1, xk1, xv1);
  }
}

__global__ void fp8_to_fp16_kernel(const uint32_t* __restrict__ in, uint2* __restrict__ out,
                                   long long n4) {
  grid_dependency_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    uint32_t lo, hi;
    e4m3x4_to_h2x2(in[i], lo, hi);
    out[i] = make_uint2(lo, hi);
  }
}

cudaError_t sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* k_new, const void* v_new, const int32_t* slots,
                                     int num_tokens, int Hkv, int D, void* k_cache,
                                     void* v_cache, long long num_slots, const float* ks,
                                     const float* vs, int per_channel, bool fp8, uint32_t* flags,
                                     cudaStream_t stream) {
  const long long ppt = (long long)Hkv * (D / 8);
  if (num_tokens == 0 || ppt == 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  // token lanes: one resident wave of CTAs in all, at most one lane per token
  long long lanes = ((long long)sms * kQuantBlocksPerSm * kQuantThreads) / ppt;
  if (lanes < 1) lanes = 1;
  if (lanes > num_tokens) lanes = num_tokens;
  const long long threads = lanes * ppt;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((threads + kQuantThreads - 1) / kQuantThreads));
  cfg.blockDim = dim3(kQuantThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kern = fp8 ? reshape_and_cache_kernel<true> : reshape_and_cache_kernel<false>;
  return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const __half*>(k_new),
                            reinterpret_cast<const __half*>(v_new), slots, num_tokens, Hkv, D,
                            static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache),
                            num_slots, ks, vs, per_channel, lanes, flags);
}

cudaError_t launch_fp8_to_fp16(const uint8_t* in, uint16_t* out, int64_t n,
                               cudaStream_t stream) {
  const long long n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  long long blocks = (n4 + 255) / 256;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  fp8_to_fp16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<const uint32_t*>(in), reinterpret_cast<uint2*>(out), n4);
  return cudaGetLastError();
}

}  // namespace i8kv
