// Split-KV GQA decode on the fifth-generation tensor cores (tcgen05, tensor
// memory) for int8 and float8 e4m3fn caches with head_dim 128 or 256.
//
// What one CTA computes is the same as the mma.sync kernel (onnxruntime PR
// 33707 "INT8-KV DynamicSparseAttention", Summary of Changes §1-§2;
// onnxruntime PR 29912 "PagedAttention", CUDA kernels): for one work unit
// (query row r, KV head g) and one split k, the G <= 16 query heads of the
// group attend the candidates at positions [k*chunk, (k+1)*chunk) of the row,
// and the CTA writes the split's partial (m, l, acc * 2^-15 * v_scale), or with
// one split the normalised output, the log-sum-exp and the head-sink rescale.
//
// Design (GB300, sm_103a):
//   * Blocks of 128 candidates.  The block is the M = 128 dimension of both
//     products (tokens on the tensor-memory lanes), so the group's heads need
//     only N = 16 (QK^T) or N = 32 (PV) columns and one accumulator serves the
//     whole CTA: there is no per-warp accumulator to merge at the end.
//   * Gathers.  A two-block ring of raw cache rows, filled with 16-byte
//     cp.async copies (row addresses from the list or block table, computed a
//     block ahead) with an XOR swizzle of the 16-byte chunks.
//   * Exact int8 -> fp16 (or e4m3fn -> fp16) conversion from the ring into
//     one shared-memory operand buffer in the MMA's core-matrix layout: first
//     K (the K-major A operand of S^T = K Q'^T), then, once that product has
//     completed, V of the same block (the MN-major A operand of
//     O^T = V^T [P_hi | P_lo]).  The two uses share one physical layout.
//   * Softmax in the natural-log domain with a running maximum per head,
//     reduced over the block's 128 tokens with a butterfly that halves the
//     head set at each exchange; the row sum stays per thread (fp32) until the
//     end.  The probability tile holds p * 2^15 as an fp16 high part and the
//     fp16 residual, side by side as 32 columns, so V is read once.
//   * O^T lives in tensor memory; when a head's maximum grows, its columns are
//     rescaled in place (tensor memory -> registers -> tensor memory) before
//     the block's PV product is issued.
//   * One thread issues the MMAs; their completion is tracked by two
//     mbarriers (QK^T done, PV done) whose waits give up after about a second
//     and flag the CTA instead of hanging.
//   * The numerical eligibility checks and the FP32 path are those of the
//     mma.sync kernel (attend_fp32).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/int8kv.h"
#include "decode_kernel.cuh"
#include "device.cuh"
#include "internal.h"
#include "tc.cuh"

namespace i8kv {

template <int D>
struct TcTile {
  static constexpr int kThreads = 256;
  static constexpr int kWarps = 8;
  static constexpr int BT = 128;                  // candidates per block (the MMA's M)
  static constexpr int kChunks = D / 16;          // 16-byte chunks of one cache row
  static constexpr int kHalfSlot = BT * D;        // the K (or V) rows of one block
  static constexpr int kSlot = 2 * kHalfSlot;
  static constexpr int kCvtOff = 2 * kSlot;       // after the two ring slots
  static constexpr int kCvtBytes = BT * D * 2;    // one block of K (or V) as fp16
  static constexpr int kPOff = kCvtOff + kCvtBytes;
  static constexpr int kPBytes = BT * 32 * 2;     // [P_hi | P_lo] of one block
  static constexpr int kQOff = kPOff + kPBytes;
  static constexpr int kQBytes = 16 * D * 2;      // Q' of 16 head slots
  static constexpr int kRowOff = kQOff + kQBytes; // long long [2][BT] row byte offsets
  static constexpr int kMaskOff = kRowOff + 2 * BT * 8;   // uint32 [2][4] valid bits
  static constexpr int kBarOff = kMaskOff + 32;   // two mbarriers
  static constexpr int kTmemSlot = kBarOff + 16;  // tensor-memory base address
  static constexpr int kRedOff = kTmemSlot + 16;  // float [4][16] exchange
  static constexpr int kVsOff = kRedOff + 4 * 16 * 4;
  static constexpr int kSmem = kVsOff + D * 4;
  // 8-token groups of a converted block are 16 * D bytes apart, 8-channel
  // groups 128 bytes (core matrix (t/8, c/8) at (t/8) * 16D + (c/8) * 128)
  static constexpr uint32_t kTokGroup = 16 * D;
  // P: core matrix (t/8, n/8) at (n/8) * 2048 + (t/8) * 128
  static constexpr uint32_t kPColGroup = (BT / 8) * 128;
  // tensor memory: S^T at columns [0, 16), O^T block cb at [32 + 32 cb, 64 + 32 cb)
  static constexpr int kOCol = 32;
  static constexpr int kCols = D == 256 ? 128 : 64;
  static_assert(D == 128 || D == 256, "head_dim");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(kRowOff % 8 == 0 && kBarOff % 8 == 0, "alignment");
};

// Convert the K (or V) rows of one ring slot (raw, 16-byte chunks XOR-swizzled
// by token) into fp16 core matrices.  Lane (t % 8, chunk % 4) mapping: the 8
// lanes of a quarter-warp read one chunk of 8 consecutive tokens (distinct
// bank groups thanks to the swizzle) and write 8 consecutive 16-byte rows of
// one core matrix.
template <int D, bool FP8>
__device__ __forceinline__ void convert_block(const uint8_t* raw, uint8_t* cvt, int warp,
                                              int lane) {
  using T = TcTile<D>;
  constexpr int kPairs = 16 * (T::kChunks / 4);  // (token group, chunk quad) pairs
  const int tl = lane & 7, cs = lane >> 3;
#pragma unroll
  for (int i = warp; i < kPairs; i += T::kWarps) {
    const int tg = i & 15, cq = i >> 4;
    const int t = 8 * tg + tl, c = 4 * cq + cs;
    const uint4 w = *reinterpret_cast<const uint4*>(raw + t * D + ((c ^ (t & 7)) << 4));
    uint32_t h[8];
    if constexpr (FP8) {
      e4m3x4_to_h2x2(w.x, h[0], h[1]);
      e4m3x4_to_h2x2(w.y, h[2], h[3]);
      e4m3x4_to_h2x2(w.z, h[4], h[5]);
      e4m3x4_to_h2x2(w.w, h[6], h[7]);
    } else {
      const uint32_t x0 = flip_i8x4(w.x), x1 = flip_i8x4(w.y);
      const uint32_t x2 = flip_i8x4(w.z), x3 = flip_i8x4(w.w);
      h[0] = i8x2_to_h2(x0, 0x4140u);
      h[1] = i8x2_to_h2(x0, 0x4342u);
      h[2] = i8x2_to_h2(x1, 0x4140u);
      h[3] = i8x2_to_h2(x1, 0x4342u);
      h[4] = i8x2_to_h2(x2, 0x4140u);
      h[5] = i8x2_to_h2(x2, 0x4342u);
      h[6] = i8x2_to_h2(x3, 0x4140u);
      h[7] = i8x2_to_h2(x3, 0x4342u);
    }
    uint8_t* dst = cvt + tg * T::kTokGroup + (2 * c) * 128 + tl * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(dst + 128) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

template <int D, bool PAGED, bool FP8>
__global__ void __launch_bounds__(256, 1) decode_tc_kernel(const DecodeParams p) {
  using T = TcTile<D>;
  constexpr int BT = T::BT;
  constexpr int kThreads = T::kThreads;
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  uint8_t* const smem = tc_smem;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int quad = warp & 3;   // tensor-memory lane quarter: tokens / channels 32 quad + lane
  const int hh = warp >> 2;    // head half: heads 8 hh .. 8 hh + 7
  const int unit = blockIdx.x;
  const int split = blockIdx.y;
  const int row = unit / p.Hkv;
  const int g = unit - row * p.Hkv;
  const int G = p.G;
  const uint32_t sbase = smem_addr(smem);
  grid_dependency_wait();  // inputs may come from the previous kernel of the stream

  // ---------------- query pieces and key scales (8 channels per piece) ----------------
  constexpr int kQSteps = 16 * D / 8 / kThreads;
  uint4 q_raw[kQSteps];
  float4 ks_raw[kQSteps][2];
  {
    const __half* qrow = reinterpret_cast<const __half*>(p.q) + ((long long)row * p.Hq + g * G) * D;
#pragma unroll
    for (int i = 0; i < kQSteps; ++i) {
      const int e = tid + i * kThreads;
      const int h = (e * 8) / D, d0 = (e * 8) % D;
      q_raw[i] = make_uint4(0u, 0u, 0u, 0u);
      ks_raw[i][0] = ks_raw[i][1] = make_float4(1.f, 1.f, 1.f, 1.f);
      if (h < G) {
        q_raw[i] = *reinterpret_cast<const uint4*>(qrow + h * D + d0);
        if (p.per_channel) {
          ks_raw[i][0] = *reinterpret_cast<const float4*>(p.k_scale + g * D + d0);
          ks_raw[i][1] = *reinterpret_cast<const float4*>(p.k_scale + g * D + d0 + 4);
        } else {
          const float k0 = p.k_scale[0];
          ks_raw[i][0] = ks_raw[i][1] = make_float4(k0, k0, k0, k0);
        }
      }
    }
  }
  float* svs = reinterpret_cast<float*>(smem + T::kVsOff);
  bool vs_bad = false;
  for (int d = tid; d < D; d += kThreads) {
    const float v = p.per_channel ? p.v_scale[g * D + d] : p.v_scale[0];
    svs[d] = v;
    vs_bad |= !(fabsf(v) <= 3.4028235e38f);
  }

  // ---------------- candidate range of this split ----------------
  const int cap = PAGED ? p.max_blocks * p.bs : p.max_sel;
  int len = 0;
  if constexpr (PAGED) len = p.seq_lens[row];
  int wlo = 0, base = 0;
  if constexpr (PAGED) {
    if (p.window >= 0) {
      const int live = min(max(len, 0), cap);
      wlo = max(0, live - 1 - p.window);
      base = wlo & ~15;
    }
  }
  const int lo = base + split * p.chunk;
  const int nhi = min(lo + p.chunk, cap);
  const int bs_shift = p.bs_log2;
  auto block_of = [&](int pos) -> int { return bs_shift >= 0 ? pos >> bs_shift : pos / p.bs; };
  auto offset_in_block = [&](int pos) -> int {
    return bs_shift >= 0 ? pos & (p.bs - 1) : pos % p.bs;
  };
  // gather key of this thread's token of block b (threads 0 .. 127; fetched
  // against the nominal end, before the live length of a paged row is known)
  auto load_key = [&](int b) -> int {
    const int pos = lo + BT * b + tid;
    if (tid >= BT || pos >= nhi) return -1;
    if constexpr (PAGED) return __ldg(p.block_table + (long long)row * p.max_blocks + block_of(pos));
    return __ldg(p.idx + (long long)row * p.max_sel + pos);
  };
  int key0 = load_key(0), key1 = load_key(1);

  int hi = nhi;
  if constexpr (PAGED) {
    if (len > cap || len < 0) {
      if (g == 0 && split == 0 && tid == 0) flag_or(p.flags, I8KV_FLAG_LEN_CLAMPED);
      len = len < 0 ? 0 : cap;
    }
    hi = min(nhi, len);
    if (p.slots_out != nullptr && g == 0) {
      for (int t = split * kThreads + tid; t < cap; t += p.num_splits * kThreads) {
        int v = -1;
        if (t >= wlo && t < len) {
          const int blk = p.block_table[(long long)row * p.max_blocks + t / p.bs];
          v = blk * p.bs + t % p.bs;
        }
        p.slots_out[(long long)row * cap + t] = v;
      }
    }
  }
  const int npos = hi > lo ? hi - lo : 0;
  const int nblk = (npos + BT - 1) / BT;

  const long long head0 = (long long)row * p.Hq + g * G;
  if (npos == 0) {
    for (int e = tid; e < G * (p.num_splits == 1 ? D : 1); e += kThreads) {
      if (p.num_splits == 1) {
        const int h = e / D, d = e % D;
        reinterpret_cast<__half*>(p.out)[(head0 + h) * D + d] = __float2half_rn(0.f);
        if (d == 0 && p.lse != nullptr) p.lse[head0 + h] = neg_inf();
      } else {
        const long long b0 = ((long long)unit * p.num_splits + split) * G + e;
        p.ws_m[b0] = neg_inf();
        p.ws_l[b0] = 0.f;
      }
    }
    return;
  }

  // ---------------- row offsets of a block, and its copies ----------------
  const char* kbase = reinterpret_cast<const char*>(p.k);
  const char* vbase = reinterpret_cast<const char*>(p.v);
  const long long row_stride = (long long)p.Hkv * D;
  long long* rowoff = reinterpret_cast<long long*>(smem + T::kRowOff);
  uint32_t* vmask = reinterpret_cast<uint32_t*>(smem + T::kMaskOff);
  // threads 0..127: the byte offset of their token's row in block b (-1 if the
  // position is not attended) and the block's valid bits, into ring slot sl
  auto publish = [&](int b, int key, int sl) {
    if (tid >= BT) return;
    const int pos = lo + BT * b + tid;
    const bool live = pos < hi && pos >= wlo;
    long long off = -1;
    if (live) {
      if constexpr (PAGED) {
        if (key >= 0 && (long long)key < p.cache_rows)
          off = ((long long)key * p.bs + offset_in_block(pos)) * row_stride + (long long)g * D;
        else
          flag_or(p.flags, I8KV_FLAG_BAD_BLOCK);
      } else {
        if (key >= 0 && (long long)key < p.cache_rows) off = (long long)key * row_stride + (long long)g * D;
      }
    }
    rowoff[sl * BT + tid] = off;
    const unsigned bits = __ballot_sync(0xffffffffu, off >= 0);
    if (lane == 0) vmask[sl * 4 + warp] = bits;
  };
  auto issue = [&](int b, int sl) {
    if (b < nblk) {
      const uint32_t dK = sbase + sl * T::kSlot;
      const uint32_t dV = dK + T::kHalfSlot;
#pragma unroll
      for (int i = tid; i < BT * T::kChunks; i += kThreads) {
        const int t = i / T::kChunks, c = i % T::kChunks;
        const long long off = rowoff[sl * BT + t];
        const bool ok = off >= 0;
        const long long src = ok ? off + c * 16 : 0;
        const uint32_t so = t * D + ((c ^ (t & 7)) << 4);
        cp_async16(dK + so, kbase + src, ok ? 16u : 0u);
        cp_async16(dV + so, vbase + src, ok ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  publish(0, key0, 0);
  publish(1, key1, 1);
  __syncthreads();
  issue(0, 0);
  issue(1, 1);

  // ---------------- Q' = fp16(Q * k_scale) in core matrices ----------------
  // (the eligibility checks of the mma.sync kernel: a non-finite or
  // out-of-range element, a folding error beyond the budget, a non-finite
  // value scale send the CTA to the FP32 path)
  uint8_t* sq = smem + T::kQOff;
  bool use_fp32 = false, vs_big_cta = false;
  {
    constexpr float kCodeMax = FP8 ? 448.f : 128.f;
    bool bad = false, over = false;
#pragma unroll
    for (int i = 0; i < kQSteps; ++i) {
      const int e = tid + i * kThreads;
      const int h = (e * 8) / D, d0 = (e * 8) % D;
      const __half2* qh = reinterpret_cast<const __half2*>(&q_raw[i]);
      const float ks[8] = {ks_raw[i][0].x, ks_raw[i][0].y, ks_raw[i][0].z, ks_raw[i][0].w,
                           ks_raw[i][1].x, ks_raw[i][1].y, ks_raw[i][1].z, ks_raw[i][1].w};
      uint32_t w[4];
      float err = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(qh[j]);
        const float x0 = f.x * ks[2 * j], x1 = f.y * ks[2 * j + 1];
        bad |= !(fabsf(x0) <= 65504.f) || !(fabsf(x1) <= 65504.f);
        w[j] = pack_h2(x0, x1);
        const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        err += fabsf(x0 - r.x) + fabsf(x1 - r.y);
      }
      // sum over the D / 8 consecutive lanes holding this head's pieces
#pragma unroll
      for (int o = 1; o < D / 8 && o < 32; o <<= 1) err += __shfl_xor_sync(0xffffffffu, err, o);
      over |= h < G && p.sigma * kCodeMax * err > kQueryErrorBudget;
      *reinterpret_cast<uint4*>(sq + (h >> 3) * T::kTokGroup + (d0 >> 3) * 128 + (h & 7) * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (bad) flag_or(p.flags, I8KV_FLAG_QUERY_RANGE);
    use_fp32 = __syncthreads_or(bad || over || vs_bad);
    bool big = false;
#pragma unroll
    for (int d = lane; d < D; d += 32) big |= fabsf(svs[d]) > kMaxValueScale;
    vs_big_cta = __any_sync(0xffffffffu, big);
  }
  if (use_fp32) {
    cp_async_wait_all();
    __syncthreads();
    if (tid == 0) flag_or(p.flags, I8KV_FLAG_FP32_PATH);
    attend_fp32<D, PAGED, false, FP8, kThreads>(p, reinterpret_cast<float*>(smem), svs,
                                                blockIdx.x, blockIdx.y);
    return;
  }

  // ---------------- tensor memory and barriers ----------------
  const uint32_t bar_s = sbase + T::kBarOff, bar_o = bar_s + 8;
  if (warp == 0) {
    tc::tmem_alloc(sbase + T::kTmemSlot, T::kCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar_s, 1);
    tc::mbar_init(bar_o, 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(smem + T::kTmemSlot);
  const uint32_t t_lane = (uint32_t)(32 * quad) << 16;

  uint8_t* cvt = smem + T::kCvtOff;
  uint8_t* pbuf = smem + T::kPOff;
  float* red = reinterpret_cast<float*>(smem + T::kRedOff);
  const float sigma = p.sigma;
  const float softcap = p.softcap;
  const float cap_k = 2.f * kLog2e / softcap;
  constexpr uint32_t kIdQK = tc::idesc_f16(128, 16, false, false);
  constexpr uint32_t kIdPV = tc::idesc_f16(128, 32, true, true);

  float m_run[8], l_thr[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    m_run[j] = neg_inf();
    l_thr[j] = 0.f;
  }
  bool deep = false, failed = false;
  int key2 = -1;

  for (int b = 0; b < nblk; ++b) {
    const int sl = b & 1;
    key2 = load_key(b + 2);  // in flight during this block
    cp_async_wait<1>();
    bool ok = true;
    if (b > 0) ok = tc::mbar_wait(bar_o, (b - 1) & 1);  // PV of the previous block is done
    // every thread's copies of the block have landed
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc::fence_after_sync();
    // K of the block -> core matrices
    convert_block<D, FP8>(smem + sl * T::kSlot, cvt, warp, lane);
    tc::fence_smem_to_async();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const uint64_t ad = tc::smem_desc(sbase + T::kCvtOff + 256 * j, 128, T::kTokGroup);
        const uint64_t bd = tc::smem_desc(sbase + T::kQOff + 256 * j, 128, T::kTokGroup);
        tc::mma_f16(tbase, ad, bd, kIdQK, j > 0);
      }
      tc::mma_commit(bar_s);
    }
    ok = tc::mbar_wait(bar_s, b & 1);
    tc::fence_after_sync();

    // ---- scores of this thread's token for heads 8 hh .. 8 hh + 7 ----
    float s[8];
    tc::tmem_ld8(tbase + t_lane + 8 * hh, s);
    tc::tmem_wait_ld();
    const bool valid = (vmask[sl * 4 + quad] >> lane) & 1u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float x = s[j] * sigma;
      if constexpr (PAGED) {
        if (softcap > 0.f) x = soft_cap(x, softcap, cap_k);
      }
      s[j] = valid ? x : neg_inf();
    }
    // block maximum per head: butterfly over the 32 tokens of the warp that
    // keeps half of the heads at each of the first three exchanges
    float mx;
    {
      float a4[4], a2[2];
      const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float send = u16 ? s[j] : s[j + 4];
        const float keep = u16 ? s[j + 4] : s[j];
        a4[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float send = u8 ? a4[j] : a4[j + 2];
        const float keep = u8 ? a4[j + 2] : a4[j];
        a2[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
      }
      {
        const float send = u4 ? a2[0] : a2[1];
        const float keep = u4 ? a2[1] : a2[0];
        mx = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    }
    // lane holds head 8 hh + (lane >> 2): 4 * bit4 + 2 * bit3 + bit2
    if ((lane & 3) == 0) red[quad * 16 + 8 * hh + (lane >> 2)] = mx;
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    float alpha[8];
    bool grew = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int h = 8 * hh + j;
      const float bm = fmaxf(fmaxf(red[h], red[16 + h]), fmaxf(red[32 + h], red[48 + h]));
      const float mnew = fmaxf(m_run[j], bm);
      const float bse = mnew == neg_inf() ? 0.f : mnew;
      alpha[j] = fast_exp2((m_run[j] - bse) * kLog2e);
      grew |= mnew != m_run[j];
      const float pr = fast_exp2((s[j] - bse) * kLog2e);
      if (vs_big_cta) deep |= s[j] != neg_inf() && s[j] < mnew - kTailDepth;
      l_thr[j] = l_thr[j] * alpha[j] + pr;
      m_run[j] = mnew;
      s[j] = pr * kProbScale;
    }
    // [P_hi | P_lo] of this token: n-groups hh (high) and 2 + hh (low)
    {
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half a = __float2half_rn(s[2 * j]), c = __float2half_rn(s[2 * j + 1]);
        ph[j] = pack_h2(a, c);
        pl[j] = pack_h2(s[2 * j] - __half2float(a), s[2 * j + 1] - __half2float(c));
      }
      const int t = 32 * quad + lane;
      uint8_t* dst = pbuf + (t >> 3) * 128 + (t & 7) * 16;
      *reinterpret_cast<uint4*>(dst + hh * T::kPColGroup) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
      *reinterpret_cast<uint4*>(dst + (2 + hh) * T::kPColGroup) =
          make_uint4(pl[0], pl[1], pl[2], pl[3]);
    }
    // rescale O^T columns of these heads when a maximum grew (warp-uniform:
    // every lane of the warp has the same heads)
    if (b > 0 && grew) {
#pragma unroll
      for (int cb = 0; cb < D / 128; ++cb) {
        const uint32_t ta = tbase + t_lane + T::kOCol + 32 * cb + 8 * hh;
        float o[8], ol[8];
        tc::tmem_ld8(ta, o);
        tc::tmem_ld8(ta + 16, ol);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          o[j] *= alpha[j];
          ol[j] *= alpha[j];
        }
        tc::tmem_st8(ta, o);
        tc::tmem_st8(ta + 16, ol);
      }
      tc::tmem_wait_st();
    }
    // V of the block -> the same core matrices (the QK^T product has read K)
    convert_block<D, FP8>(smem + sl * T::kSlot + T::kHalfSlot, cvt, warp, lane);
    // row offsets of block b + 2 into this ring slot (its copies start below)
    publish(b + 2, key2, sl);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int cb = 0; cb < D / 128; ++cb) {
#pragma unroll
        for (int j = 0; j < BT / 16; ++j) {
          const uint64_t ad = tc::smem_desc(sbase + T::kCvtOff + cb * 2048 + 2 * j * T::kTokGroup,
                                            T::kTokGroup, 128);
          const uint64_t bd = tc::smem_desc(sbase + T::kPOff + 256 * j, 128, T::kPColGroup);
          tc::mma_f16(tbase + T::kOCol + 32 * cb, ad, bd, kIdPV, b > 0 || j > 0);
        }
      }
      tc::mma_commit(bar_o);
    }
    issue(b + 2, sl);
  }

  if (!failed) {
    failed = !tc::mbar_wait(bar_o, (nblk - 1) & 1);
    tc::fence_after_sync();
    failed = __syncthreads_or(failed);
  }
  cp_async_wait_all();
  if (failed) {
    if (tid == 0) flag_or(p.flags, I8KV_FLAG_WAIT_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, T::kCols);
    return;
  }

  // a large value scale with a deep candidate: start over on the FP32 path
  if (vs_big_cta && __syncthreads_or(deep)) {
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, T::kCols);
    if (tid == 0) flag_or(p.flags, I8KV_FLAG_FP32_PATH);
    attend_fp32<D, PAGED, false, FP8, kThreads>(p, reinterpret_cast<float*>(smem), svs,
                                                blockIdx.x, blockIdx.y);
    return;
  }

  // ---------------- row sums: butterfly over the warp, then the 4 quarters ----------------
  {
    float a4[4], a2[2], sm;
    const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = u16 ? l_thr[j] : l_thr[j + 4];
      const float keep = u16 ? l_thr[j + 4] : l_thr[j];
      a4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float send = u8 ? a4[j] : a4[j + 2];
      const float keep = u8 ? a4[j + 2] : a4[j];
      a2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    {
      const float send = u4 ? a2[0] : a2[1];
      const float keep = u4 ? a2[1] : a2[0];
      sm = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    sm += __shfl_xor_sync(0xffffffffu, sm, 2);
    sm += __shfl_xor_sync(0xffffffffu, sm, 1);
    __syncthreads();  // the block maxima in `red` have been read
    if ((lane & 3) == 0) red[quad * 16 + 8 * hh + (lane >> 2)] = sm;
    __syncthreads();
  }

  // ---------------- epilogue: O^T columns of this thread's channel and heads ----------------
  const bool direct = p.num_splits == 1;
  float L[8], sc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int h = 8 * hh + j;
    L[j] = red[h] + red[16 + h] + red[32 + h] + red[48 + h];
    sc[j] = 0.f;
    if (L[j] > 0.f) {
      if (direct) {
        sc[j] = kInvProbScale / L[j];
        if (p.sink != nullptr && h < G)
          sc[j] *= 1.f / (1.f + expf(p.sink[g * G + h] - (m_run[j] + logf(L[j]))));
      } else {
        sc[j] = kInvProbScale;
      }
    }
  }
#pragma unroll
  for (int cb = 0; cb < D / 128; ++cb) {
    const uint32_t ta = tbase + t_lane + T::kOCol + 32 * cb + 8 * hh;
    float o[8], ol[8];
    tc::tmem_ld8(ta, o);
    tc::tmem_ld8(ta + 16, ol);
    tc::tmem_wait_ld();
    const int d = 128 * cb + 32 * quad + lane;
    const float vs = svs[d];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int h = 8 * hh + j;
      if (h >= G) continue;
      const float val = (o[j] + ol[j]) * sc[j] * vs;
      if (direct) {
        reinterpret_cast<__half*>(p.out)[(head0 + h) * D + d] = __float2half_rn(val);
      } else if (L[j] > 0.f) {
        const long long b0 = ((long long)unit * p.num_splits + split) * G + h;
        p.ws_acc[b0 * D + d] = val;
      }
    }
  }
  if (quad == 0 && lane < 8) {
    const int h = 8 * hh + lane;
    if (h < G) {
      float Lh = 0.f, Mh = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j == lane) {
          Lh = L[j];
          Mh = m_run[j];
        }
      if (direct) {
        if (p.lse != nullptr) p.lse[head0 + h] = Lh > 0.f ? Mh + logf(Lh) : neg_inf();
      } else {
        const long long b0 = ((long long)unit * p.num_splits + split) * G + h;
        p.ws_m[b0] = Lh > 0.f ? Mh : neg_inf();
        p.ws_l[b0] = Lh;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, T::kCols);
}

template <int D, bool PAGED, bool FP8>
cudaError_t run_decode_tc(const DecodeParams& p, cudaStream_t s, int* occupancy) {
  using T = TcTile<D>;
  auto kern = decode_tc_kernel<D, PAGED, FP8>;
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(done.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  if (occupancy != nullptr) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, kern, T::kThreads, T::kSmem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.rows * p.Hkv), (unsigned)p.num_splits);
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

// The tensor-memory kernel serves int8 / e4m3fn caches with head_dim 128 or
// 256 and up to 16 query heads per KV head; everything else stays on the
// mma.sync kernel.
template <bool PAGED, bool FP8>
cudaError_t dispatch_decode_tc(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                               int* occupancy) {
  switch (key.D) {
    case 128: return run_decode_tc<128, PAGED, FP8>(p, s, occupancy);
    case 256: return run_decode_tc<256, PAGED, FP8>(p, s, occupancy);
    default: return dispatch_decode<PAGED, false, true, FP8>(key, p, s, occupancy);
  }
}

}  // namespace i8kv
