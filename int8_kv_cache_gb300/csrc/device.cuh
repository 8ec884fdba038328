// Device helpers shared by the decode / prefill / combine kernels: inline PTX
// for asynchronous copies, shared-memory matrix loads, warp matrix transposes,
// FP16 tensor-core MMA and the exact int8 -> fp16 conversion.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace i8kv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kProbScale = 32768.0f;        // probability tile holds p * 2^15
constexpr float kInvProbScale = 1.0f / 32768.0f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x with the SFU instruction (relative error about 2^-22; 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// 1/x with the SFU instruction (relative error about 2^-23; 1/inf = +0).
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Softcap c * tanh(x / c) through the identity tanh(y) = 1 - 2 / (1 + e^(2y)),
// with k = 2 log2(e) / c: e^(2y) = 2^(k x).  Saturates to +-c (2^(k x) = inf or
// 0); the absolute error is a few ulp of c, and the map has slope <= 1, so it
// never enlarges an error already in x.
__device__ __forceinline__ float soft_cap(float x, float c, float k) {
  const float e = fast_exp2(x * k);
  return fmaf(-2.f * c, fast_rcp(1.f + e), c);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global -> shared copy that bypasses L1.  src_bytes = 0
// reads nothing and zero-fills the 16 destination bytes.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// Four 8x8 b16 matrices from shared memory (lane i gives row i%8 of matrix i/8).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Same, each matrix transposed on the way.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Transpose an 8x8 b16 matrix held in the warp's registers.
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Exact int8 -> fp16 for two bytes of a word whose bytes were XOR-ed with 0x80.
// The selected byte u = code + 128 becomes the low mantissa byte of an fp16
// whose high byte is 0x64, i.e. the value 1024 + u = 1152 + code; subtracting
// 1152 (bit pattern 0x6480) is exact.  `sel` picks the two bytes:
//   0x4140: bytes 0,1   0x4342: bytes 2,3   0x4240: bytes 0,2   0x4341: bytes 1,3
// (low half of the result = first byte).
__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t xflipped, uint32_t sel) {
  uint32_t h = prmt(xflipped, 0x64646464u, sel);
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(h), "r"(0x64806480u));
  return r;
}
__device__ __forceinline__ uint32_t flip_i8x4(uint32_t w) { return w ^ 0x80808080u; }

// Four float8 e4m3fn values (bytes b0..b3 of w) -> half2 (b0, b1) and half2
// (b2, b3), with the hardware conversion (exact: every e4m3fn value is an fp16
// value; the two NaN patterns give NaN).
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  __half2 h = __halves2half2(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Programmatic dependent launch: wait until the preceding grid of the stream
// has completed and its writes are visible (returns at once when the kernel
// was launched without the programmatic-serialization attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// No kernel here lets its dependents launch early (griddepcontrol.
// launch_dependents): measured on graphs of decode calls, an early trigger at
// decode entry made the calls slower, and one at combine entry took the sparse
// decode (S = 8) from 11.53 to 11.22 us per call but the ragged paged decode
// from 37.3 to 40.8 us.

__device__ __forceinline__ void flag_or(uint32_t* flags, uint32_t bits) {
  if (flags != nullptr) atomicOr(flags, bits);
}

}  // namespace i8kv
