// Split-KV GQA decode / prefill kernel over an INT8 (or FP16) KV cache.
//
// What one CTA computes (onnxruntime PR 33707 "INT8-KV DynamicSparseAttention",
// Summary of Changes §1-§2; onnxruntime PR 29912 "PagedAttention", CUDA
// kernels): for one work unit (query row r, KV head g) and one split k, the G
// query heads of the group attend the candidates at positions
// [k*chunk, (k+1)*chunk) of the row (list positions of a sparse index list, or
// token positions of a paged sequence).  It either writes the un-normalised
// partial (m, l, acc * 2^-15 * v_scale) of the split, or, with one split, the
// normalised output, the log-sum-exp and the head-sink rescale.
//
// Design (GB300, sm_103a, 128 threads = 4 warps per CTA):
//   * Warp-private pipelines.  Warp w owns the 16-token slices w, w+4, w+8, ...
//     of the split.  It gathers each slice's K and V rows with 16-byte
//     cp.async copies into its own shared-memory ring (kStages deep), so its
//     loads stay in flight while it computes earlier slices, and it runs its
//     own online softmax.  The warps meet once, at the end, to merge their
//     (m, l, acc) through shared memory.  No warp waits on another in the loop.
//   * Tensor cores.  QK^T is S^T[token][head] = K[token][d] * Q'[head][d]^T
//     with tokens as the M=16 dimension and the group's query heads as N (8 per
//     tile, G <= 8 -> 1 tile, G <= 16 -> 2): mma.sync m16n8k16 f16 x f16 -> f32.
//     PV is O^T[d][head] = V^T[d][token] * P^T[token][head] with d as M.  The
//     probability fragments come from the QK accumulators through a warp
//     transpose (movmatrix), V^T fragments from ldmatrix.trans.
//   * Exact int8 -> fp16 in registers: each 32-bit word of codes is XOR-ed with
//     0x80808080, two bytes are permuted into the mantissa of 0x64xx
//     (= 1152 + code) and 1152 is subtracted with one fp16x2 instruction; the K
//     fragments use a permuted contraction order (4 consecutive channels per
//     thread), the V fragments take byte pairs straight from ldmatrix.trans.
//   * Numerics of the pages: k_scale is folded into the query once per CTA
//     (Q' = fp16(Q * k_scale)); scores and the running maximum stay in natural
//     log units and only (s - m) is scaled by log2(e) for exp2; the row sum is
//     unscaled fp32; the probability tile holds p * 2^15 as fp16, for decode as
//     a high part plus the fp16 residual; value_scale is applied once at the
//     end, after the accumulator has been divided by 2^15 (PR 33707 §1-§2,
//     Numerics).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/int8kv.h"
#include "device.cuh"
#include "internal.h"

namespace i8kv {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kSlice = 16;  // tokens per warp step (the MMA M dimension)

template <int D, bool FP16C>
struct Tile {
  static constexpr int kElem = FP16C ? 2 : 1;
  static constexpr int kRowBytes = D * kElem;        // one cache row of one KV head
  static constexpr int kRS = kRowBytes + 16;         // padded shared-memory row stride
  static constexpr int kChunks = kRowBytes / 16;     // 16-byte chunks per row (<= 32)
  static constexpr int kRowsPerCopy = 32 / kChunks;  // rows covered by one warp-wide copy
  static constexpr int kCopies = kSlice / kRowsPerCopy;
  static constexpr int kSliceBytes = kSlice * kRS;   // K (or V) of one slice
  static constexpr int kStages = kRowBytes <= 128 ? 4 : 3;
  static constexpr int kWarpRing = kStages * 2 * kSliceBytes;
  static constexpr int kRingBytes = kWarps * kWarpRing;
  static constexpr int kMaskBytes = kWarps * kStages * 4;
  static constexpr int kQBytes = 16 * D * 2;         // Q' staging, 16 heads x D fp16
  static constexpr int kLoopBytes = kRingBytes + kMaskBytes + kQBytes;
  // end-of-CTA merge: m, l [4][16]; acc [4][16][D]; weights [4][16]; M, L [16]
  static constexpr int kMergeBytes = (64 + 64 + kWarps * 16 * D + 64 + 16 + 16) * 4;
  static constexpr int kSmem = kLoopBytes > kMergeBytes ? kLoopBytes : kMergeBytes;
  static_assert(kChunks <= 32 && 32 % kChunks == 0, "row layout");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

template <int D, int NT, bool PAGED, bool FP16C, bool PLO>
__global__ void __launch_bounds__(kThreads, 1)
decode_kernel(const DecodeParams p) {
  using T = Tile<D, FP16C>;
  constexpr int KC = D / 16;  // k-chunks of QK^T and m-tiles of PV
  extern __shared__ __align__(128) uint8_t smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int grp = lane >> 2;
  const int tig = lane & 3;
  const int unit = blockIdx.x;
  const int split = blockIdx.y;
  const int row = unit / p.Hkv;
  const int g = unit - row * p.Hkv;
  const int G = p.G;

  // ---------------- candidate range of this split ----------------
  const long long lo = (long long)split * p.chunk;
  long long hi;
  int live = 0;
  if constexpr (PAGED) {
    const int cap = p.max_blocks * p.bs;
    int len = p.seq_lens[row];
    if (len > cap || len < 0) {
      if (g == 0 && split == 0 && threadIdx.x == 0) flag_or(p.flags, I8KV_FLAG_LEN_CLAMPED);
      len = len < 0 ? 0 : cap;
    }
    live = len;
    hi = lo + p.chunk < (long long)len ? lo + p.chunk : (long long)len;
    // debug output: the gathered row of every token of this split's nominal range
    if (p.slots_out != nullptr && g == 0) {
      const long long nhi = lo + p.chunk < (long long)cap ? lo + p.chunk : (long long)cap;
      for (long long t = lo + threadIdx.x; t < nhi; t += kThreads) {
        int v = -1;
        if (t < live) {
          const int blk = p.block_table[(long long)row * p.max_blocks + t / p.bs];
          v = blk * p.bs + (int)(t % p.bs);
        }
        p.slots_out[(long long)row * cap + t] = v;
      }
    }
  } else {
    hi = lo + p.chunk < (long long)p.max_sel ? lo + p.chunk : (long long)p.max_sel;
  }
  const int npos = hi > lo ? (int)(hi - lo) : 0;

  // ---------------- Q' = fp16(Q * k_scale), staged through shared memory ----------------
  __half* sq = reinterpret_cast<__half*>(smem + T::kRingBytes + T::kMaskBytes);
  {
    const __half* qrow = reinterpret_cast<const __half*>(p.q) + ((long long)row * p.Hq + g * G) * D;
    bool bad = false;
    for (int e = threadIdx.x; e < 8 * NT * D; e += kThreads) {
      const int h = e / D, d = e - (e / D) * D;
      float x = 0.f;
      if (h < G) {
        x = __half2float(qrow[h * D + d]);
        if constexpr (!FP16C) {
          const float ks = p.per_channel ? p.k_scale[g * D + d] : p.k_scale[0];
          x *= ks;
          bad |= !(fabsf(x) <= 65504.f);
        }
      }
      sq[h * D + d] = __float2half_rn(x);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_or(p.flags, I8KV_FLAG_QUERY_RANGE);
  }
  // B fragments of Q'^T (k = channel, n = head) in the contraction order of the
  // K fragments: int8 caches take channels 16kc + 4tig + {0,1} / {2,3}, fp16
  // caches the natural 16kc + 2tig + {0,1} / {8,9}.
  uint32_t qf[NT][KC][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(sq + (nt * 8 + grp) * D);
#pragma unroll
    for (int kc = 0; kc < KC; ++kc) {
      if constexpr (FP16C) {
        qf[nt][kc][0] = qw[(16 * kc + 2 * tig) / 2];
        qf[nt][kc][1] = qw[(16 * kc + 2 * tig + 8) / 2];
      } else {
        qf[nt][kc][0] = qw[(16 * kc + 4 * tig) / 2];
        qf[nt][kc][1] = qw[(16 * kc + 4 * tig + 2) / 2];
      }
    }
  }

  // ---------------- per-warp gather pipeline ----------------
  const int nslices = (npos + kSlice - 1) / kSlice;
  const int my_n = nslices > warp ? (nslices - warp + kWarps - 1) / kWarps : 0;
  uint8_t* wring = smem + warp * T::kWarpRing;
  int* wmask = reinterpret_cast<int*>(smem + T::kRingBytes) + warp * T::kStages;
  const uint32_t ring_addr = smem_addr(wring);

  const char* kbase = reinterpret_cast<const char*>(p.k);
  const char* vbase = reinterpret_cast<const char*>(p.v);
  const long long row_stride = (long long)p.Hkv * T::kRowBytes;  // bytes between tokens
  const int chunk_id = lane % T::kChunks;
  const int row_in_copy = lane / T::kChunks;
  const long long lane_off = (long long)g * T::kRowBytes + chunk_id * 16;

  auto slice_pos = [&](int k) -> long long { return lo + (long long)kSlice * (warp + kWarps * k); };

  // The per-slice gather key, loaded ahead of the copies: the list entry of
  // row (lane & 15) of the slice (sparse), or the block id (paged).
  auto fetch = [&](int k) -> int {
    if (k >= my_n) return -1;
    const long long pos0 = slice_pos(k);
    if constexpr (PAGED) {
      return __ldg(p.block_table + (long long)row * p.max_blocks + pos0 / p.bs);
    } else {
      const long long pos = pos0 + (lane & 15);
      return pos < hi ? __ldg(p.idx + (long long)row * p.max_sel + pos) : -1;
    }
  };

  auto issue = [&](int k, int key) {
    if (k < my_n) {
      const long long pos0 = slice_pos(k);
      const int st = k % T::kStages;
      const uint32_t dK = ring_addr + st * 2 * T::kSliceBytes;
      const uint32_t dV = dK + T::kSliceBytes;
      int mask;
      if constexpr (PAGED) {
        int nvalid = hi - pos0 < kSlice ? (int)(hi - pos0) : kSlice;
        if (key < 0 || (long long)key >= p.cache_rows) {
          if (lane == 0) flag_or(p.flags, I8KV_FLAG_BAD_BLOCK);
          nvalid = 0;
        }
        mask = nvalid >= kSlice ? 0xFFFF : ((1 << nvalid) - 1);
        const long long rbase = (long long)key * p.bs + (pos0 % p.bs);
#pragma unroll
        for (int i = 0; i < T::kCopies; ++i) {
          const int r = row_in_copy + i * T::kRowsPerCopy;
          const bool ok = r < nvalid;
          const long long off = ok ? (rbase + r) * row_stride + lane_off : 0;
          cp_async16(dK + r * T::kRS + chunk_id * 16, kbase + off, ok ? 16u : 0u);
          cp_async16(dV + r * T::kRS + chunk_id * 16, vbase + off, ok ? 16u : 0u);
        }
      } else {
        const bool ok_mine = key >= 0 && (long long)key < p.cache_rows;
        mask = (int)(__ballot_sync(0xffffffffu, ok_mine) & 0xFFFFu);
#pragma unroll
        for (int i = 0; i < T::kCopies; ++i) {
          const int r = row_in_copy + i * T::kRowsPerCopy;
          const int t = __shfl_sync(0xffffffffu, key, r);
          const bool ok = (mask >> r) & 1;
          const long long off = ok ? (long long)t * row_stride + lane_off : 0;
          cp_async16(dK + r * T::kRS + chunk_id * 16, kbase + off, ok ? 16u : 0u);
          cp_async16(dV + r * T::kRS + chunk_id * 16, vbase + off, ok ? 16u : 0u);
        }
      }
      if (lane == 0) wmask[st] = mask;
    }
    cp_async_commit();
  };

  // accumulators: O^T m-tiles [KC][NT][4]; online-softmax state per (nt, head pair)
  float acc[KC][NT][4];
  float mrun[NT][2], lrun[NT][2];
#pragma unroll
  for (int mt = 0; mt < KC; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mrun[nt][0] = mrun[nt][1] = neg_inf();
    lrun[nt][0] = lrun[nt][1] = 0.f;
  }

  // ldmatrix lane address: matrix m = lane/8 covers tokens (lane%8) + 8*(m&1)
  // of 16-byte chunk (m>>1) (+ 2 per step)
  const uint32_t ld_off = ((lane & 7) + 8 * ((lane >> 3) & 1)) * T::kRS + (lane >> 4) * 16;
  const float sigma = p.sigma;

  {
    int pf[T::kStages + 1];
#pragma unroll
    for (int k = 0; k <= T::kStages; ++k) pf[k] = fetch(k);
#pragma unroll
    for (int k = 0; k < T::kStages - 1; ++k) issue(k, pf[k]);
    int q0 = pf[T::kStages - 1], q1 = pf[T::kStages];

    for (int k = 0; k < my_n; ++k) {
      issue(k + T::kStages - 1, q0);
      q0 = q1;
      q1 = fetch(k + T::kStages + 1);
      cp_async_wait<T::kStages - 1>();
      __syncwarp();

      const int st = k % T::kStages;
      const uint32_t sK = ring_addr + st * 2 * T::kSliceBytes;
      const uint32_t sV = sK + T::kSliceBytes;
      const int mask = wmask[st];

      // ---- S^T = K Q'^T ----
      float sacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
      for (int c2 = 0; c2 < T::kChunks / 2; ++c2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(sK + ld_off + 32 * c2, r0, r1, r2, r3);
        if constexpr (FP16C) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma16816(sacc[nt], r0, r1, r2, r3, qf[nt][c2][0], qf[nt][c2][1]);
        } else {
          const uint32_t x0 = flip_i8x4(r0), x1 = flip_i8x4(r1);
          const uint32_t x2 = flip_i8x4(r2), x3 = flip_i8x4(r3);
          {
            const uint32_t a0 = i8x2_to_h2(x0, 0x4140u), a1 = i8x2_to_h2(x1, 0x4140u);
            const uint32_t a2 = i8x2_to_h2(x0, 0x4342u), a3 = i8x2_to_h2(x1, 0x4342u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816(sacc[nt], a0, a1, a2, a3, qf[nt][2 * c2][0], qf[nt][2 * c2][1]);
          }
          {
            const uint32_t a0 = i8x2_to_h2(x2, 0x4140u), a1 = i8x2_to_h2(x3, 0x4140u);
            const uint32_t a2 = i8x2_to_h2(x2, 0x4342u), a3 = i8x2_to_h2(x3, 0x4342u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816(sacc[nt], a0, a1, a2, a3, qf[nt][2 * c2 + 1][0], qf[nt][2 * c2 + 1][1]);
          }
        }
      }

      // ---- online softmax (natural log domain) and the probability tile ----
      const bool v_top = (mask >> grp) & 1;
      const bool v_bot = (mask >> (grp + 8)) & 1;
      uint32_t ph[NT][2], pl[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float s[4];
        s[0] = v_top ? sacc[nt][0] * sigma : neg_inf();
        s[1] = v_top ? sacc[nt][1] * sigma : neg_inf();
        s[2] = v_bot ? sacc[nt][2] * sigma : neg_inf();
        s[3] = v_bot ? sacc[nt][3] * sigma : neg_inf();
        float pr[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // head 2*tig + j of this n-tile
          float mx = fmaxf(s[j], s[2 + j]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(mrun[nt][j], mx);
          const float base = mnew == neg_inf() ? 0.f : mnew;
          const float alpha = fast_exp2((mrun[nt][j] - base) * kLog2e);
          pr[j] = fast_exp2((s[j] - base) * kLog2e);
          pr[2 + j] = fast_exp2((s[2 + j] - base) * kLog2e);
          lrun[nt][j] = lrun[nt][j] * alpha + pr[j] + pr[2 + j];
          mrun[nt][j] = mnew;
#pragma unroll
          for (int mt = 0; mt < KC; ++mt) {
            acc[mt][nt][j] *= alpha;
            acc[mt][nt][2 + j] *= alpha;
          }
        }
        __half hh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) hh[e] = __float2half_rn(pr[e] * kProbScale);
        ph[nt][0] = movm_t(pack_h2(hh[0], hh[1]));
        ph[nt][1] = movm_t(pack_h2(hh[2], hh[3]));
        if constexpr (PLO) {
          __half hl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) hl[e] = __float2half_rn(pr[e] * kProbScale - __half2float(hh[e]));
          pl[nt][0] = movm_t(pack_h2(hl[0], hl[1]));
          pl[nt][1] = movm_t(pack_h2(hl[2], hl[3]));
        }
      }

      // ---- O^T += V^T P^T ----
#pragma unroll
      for (int c2 = 0; c2 < T::kChunks / 2; ++c2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(sV + ld_off + 32 * c2, r0, r1, r2, r3);
        if constexpr (FP16C) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(acc[c2][nt], r0, r2, r1, r3, ph[nt][0], ph[nt][1]);
            if constexpr (PLO) mma16816(acc[c2][nt], r0, r2, r1, r3, pl[nt][0], pl[nt][1]);
          }
        } else {
          const uint32_t x0 = flip_i8x4(r0), x1 = flip_i8x4(r1);
          const uint32_t x2 = flip_i8x4(r2), x3 = flip_i8x4(r3);
          {
            const uint32_t a0 = i8x2_to_h2(x0, 0x4240u), a1 = i8x2_to_h2(x0, 0x4341u);
            const uint32_t a2 = i8x2_to_h2(x1, 0x4240u), a3 = i8x2_to_h2(x1, 0x4341u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma16816(acc[2 * c2][nt], a0, a1, a2, a3, ph[nt][0], ph[nt][1]);
              if constexpr (PLO) mma16816(acc[2 * c2][nt], a0, a1, a2, a3, pl[nt][0], pl[nt][1]);
            }
          }
          {
            const uint32_t a0 = i8x2_to_h2(x2, 0x4240u), a1 = i8x2_to_h2(x2, 0x4341u);
            const uint32_t a2 = i8x2_to_h2(x3, 0x4240u), a3 = i8x2_to_h2(x3, 0x4341u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma16816(acc[2 * c2 + 1][nt], a0, a1, a2, a3, ph[nt][0], ph[nt][1]);
              if constexpr (PLO)
                mma16816(acc[2 * c2 + 1][nt], a0, a1, a2, a3, pl[nt][0], pl[nt][1]);
            }
          }
        }
      }
      __syncwarp();
    }
  }
  cp_async_wait_all();
  __syncthreads();  // every warp is done with its ring: reuse the memory for the merge

  // ---------------- merge the four warps' partials ----------------
  float* mw = reinterpret_cast<float*>(smem);  // [4][16]
  float* lw = mw + 64;                         // [4][16]
  float* aw = lw + 64;                         // [4][16][D]
  float* fw = aw + kWarps * 16 * D;            // [4][16]
  float* Ms = fw + 64;                         // [16]
  float* Ls = Ms + 16;                         // [16]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = lrun[nt][j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (grp == 0) {
        mw[warp * 16 + nt * 8 + 2 * tig + j] = mrun[nt][j];
        lw[warp * 16 + nt * 8 + 2 * tig + j] = l;
      }
    }
#pragma unroll
    for (int mt = 0; mt < KC; ++mt) {
      const int h = nt * 8 + 2 * tig;
      int da, db;
      if constexpr (FP16C) {
        da = 16 * mt + grp;
        db = da + 8;
      } else {
        da = 16 * mt + 2 * grp;
        db = da + 1;
      }
      float* a0 = aw + (warp * 16 + h) * D;
      float* a1 = a0 + D;
      a0[da] = acc[mt][nt][0];
      a0[db] = acc[mt][nt][2];
      a1[da] = acc[mt][nt][1];
      a1[db] = acc[mt][nt][3];
    }
  }
  if (NT == 1) {  // heads 8..15 of the merge area are never written: keep them inert
    for (int e = threadIdx.x; e < kWarps * 8; e += kThreads) {
      mw[(e / 8) * 16 + 8 + (e % 8)] = neg_inf();
      lw[(e / 8) * 16 + 8 + (e % 8)] = 0.f;
    }
  }
  __syncthreads();
  if (threadIdx.x < 16) {
    const int h = threadIdx.x;
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * 16 + h]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = M == neg_inf() ? 0.f : fast_exp2((mw[w * 16 + h] - M) * kLog2e);
      fw[w * 16 + h] = f;
      L += f * lw[w * 16 + h];
    }
    Ms[h] = M;
    Ls[h] = L;
  }
  __syncthreads();

  const bool direct = p.num_splits == 1;
  const long long out_head0 = (long long)row * p.Hq + g * G;
  for (int e = threadIdx.x; e < G * D; e += kThreads) {
    const int h = e / D, d = e - (e / D) * D;
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) a += fw[w * 16 + h] * aw[(w * 16 + h) * D + d];
    float vs = 1.f;
    if constexpr (!FP16C) vs = p.per_channel ? p.v_scale[g * D + d] : p.v_scale[0];
    const float M = Ms[h], L = Ls[h];
    if (direct) {
      float o = 0.f;
      float lse = neg_inf();
      if (L > 0.f) {
        lse = M + logf(L);
        o = (a * kInvProbScale / L) * vs;
        if (p.sink != nullptr) o *= 1.f / (1.f + expf(p.sink[g * G + h] - lse));
      }
      reinterpret_cast<__half*>(p.out)[(out_head0 + h) * D + d] = __float2half_rn(o);
      if (d == 0 && p.lse != nullptr) p.lse[out_head0 + h] = lse;
    } else {
      const long long base = ((long long)unit * p.num_splits + split) * G + h;
      if (L > 0.f) p.ws_acc[base * D + d] = (a * kInvProbScale) * vs;
      if (d == 0) {
        p.ws_m[base] = L > 0.f ? M : neg_inf();
        p.ws_l[base] = L;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host-side launch of one instantiation
// ---------------------------------------------------------------------------

template <int D, int NT, bool PAGED, bool FP16C, bool PLO>
cudaError_t run_decode(const DecodeParams& p, cudaStream_t s, int* occupancy) {
  using T = Tile<D, FP16C>;
  auto kern = decode_kernel<D, NT, PAGED, FP16C, PLO>;
  // the opt-in shared-memory size is a per-function attribute: set it once per device
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(done.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  if (occupancy != nullptr) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, kern, kThreads, T::kSmem);
  }
  const dim3 grid((unsigned)(p.rows * p.Hkv), (unsigned)p.num_splits);
  kern<<<grid, kThreads, T::kSmem, s>>>(p);
  return cudaGetLastError();
}

template <bool PAGED, bool FP16C, bool PLO>
cudaError_t dispatch_decode(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                            int* occupancy) {
  switch (key.D * 10 + key.nt) {
    case 641: return run_decode<64, 1, PAGED, FP16C, PLO>(p, s, occupancy);
    case 642: return run_decode<64, 2, PAGED, FP16C, PLO>(p, s, occupancy);
    case 1281: return run_decode<128, 1, PAGED, FP16C, PLO>(p, s, occupancy);
    case 1282: return run_decode<128, 2, PAGED, FP16C, PLO>(p, s, occupancy);
    case 2561: return run_decode<256, 1, PAGED, FP16C, PLO>(p, s, occupancy);
    case 2562: return run_decode<256, 2, PAGED, FP16C, PLO>(p, s, occupancy);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace i8kv
