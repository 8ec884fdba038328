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
// Design (GB300, sm_103a):
//   * CTA shape.  The sparse-candidate kernel runs one CTA per SM of 4 to 16
//     warps (as many 4-warp groups as the registers and shared memory allow);
//     the paged kernel runs 4-warp CTAs, 2 to 4 per SM, so that the splits of
//     sequences of very different lengths spread over the SMs.
//   * Dispatch order (paged, long chunks).  A CTA may take another (unit,
//     split) item than its grid position names, so that the longest chunks of
//     a ragged batch start first (lpt_item below); the geometry is unchanged.
//   * Balanced pieces (paged, chunk 0 on the API).  The grid and the partial
//     slots still follow the arguments, but each CTA cuts its own piece of a
//     row's live range from all live lengths, so that a ragged batch's pieces
//     come out about equally long (balanced_item below).
//   * Warp-private pipelines.  Warp w owns the steps w, w + kWarps, ... of the
//     split (a step is 16 tokens, or 32 when two tiles fit the registers).  It
//     gathers each step's K and V rows with 16-byte cp.async copies into its
//     own shared-memory ring (2 to 4 stages), so its loads stay in flight while
//     it computes earlier steps, and it runs its own online softmax.  The warps
//     meet once, at the end, to merge their (m, l, acc) through shared memory.
//     No warp waits on another in the loop.
//   * Numerical eligibility.  A CTA whose FP16 rounding cannot be bounded
//     (query folding beyond the budget, a non-finite value scale, a large value
//     scale with a deep tail) evaluates its heads on the FP32 path instead.
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
#include <type_traits>
#include <cuda_runtime.h>


#include "../../include/int8kv.h"
#include "device.cuh"
#include "internal.h"

namespace i8kv {

constexpr int kSub = 16;  // tokens per MMA tile (the M dimension of QK^T)

// SMALL: 4-warp CTAs, several per SM (the paged kernel, and the gathering
// prefill: many units, no splits); else one CTA per SM with all the warps
// that fit (the sparse decode's short splits).
template <int D, int NT, bool FP16C, bool SMALL>
struct Tile {
  static constexpr int kElem = FP16C ? 2 : 1;
  static constexpr int kRowBytes = D * kElem;        // one cache row of one KV head
  static constexpr int kChunks = kRowBytes / 16;     // 16-byte chunks per row (<= 32)
  // Tokens per warp step: two 16-token tiles where the registers allow it.
  static constexpr int SUB = (kRowBytes <= 128 && D * NT <= 256) ? 2 : 1;
  static constexpr int kStep = kSub * SUB;
  static constexpr int kRowsPerCopy = 32 / kChunks;  // rows covered by one warp-wide copy
  static constexpr int kCopies = kStep / kRowsPerCopy;
  static constexpr int kTileBytes = kStep * kRowBytes;   // K (or V) of one step, dense
  static constexpr int kStageBytes = 2 * kTileBytes;
  // Q' staging row (halves), padded so that the B-fragment loads of a warp
  // fall in distinct banks: 4-byte loads (fp16 cache) want a row offset of 4
  // banks, 8-byte loads (int8 / e4m3fn: 4 channels per thread) 8 banks
  static constexpr int kQStride = FP16C ? D + 8 : D + 16;
  static constexpr int kQBytes = 16 * kQStride * 2;
  // 4-warp groups per SM the registers allow (16, 12 or 8 warps per SM) ...
  static constexpr int kRegGroups = D * NT >= 512 ? 2 : (D * NT >= 256 ? 3 : 4);
  static constexpr int kPerGroup = 227 * 1024 / kRegGroups - 1024 - kQBytes - 256;
  // ... the ring depth per warp: the largest of 4, 3, 2 stages that fits ...
  static constexpr int kStages = 4 * 4 * kStageBytes <= kPerGroup ? 4
                               : (4 * 3 * kStageBytes <= kPerGroup ? 3 : 2);
  static constexpr int kWarpRing = kStages * kStageBytes;
  // ... and the CTA shape: the sparse-candidate decode puts them all in one
  // CTA per SM (4 to 16 warps: fewer, larger CTAs for its short splits); the
  // paged kernel keeps 4-warp CTAs, several per SM, so that the splits of
  // sequences of very different lengths spread more evenly over the SMs, and
  // so does the gathering prefill (thousands of unsplit units: one CTA's
  // prologue and merge overlap another's streaming).
  static constexpr int kSmemGroups = (227 * 1024 - 1024 - kQBytes - 256) / (4 * kWarpRing);
  static constexpr int kFitGroups = kSmemGroups < kRegGroups ? kSmemGroups : kRegGroups;
  static constexpr int kGroups = SMALL ? 1 : kFitGroups;
  static constexpr int kWarps = 4 * kGroups;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kMaskBytes = kWarps * 4 * 4;
  static constexpr int kRingBytes = kWarps * kWarpRing;
  static constexpr int kLoopBytes = kRingBytes + kMaskBytes + kQBytes;
  // end-of-CTA merge: each warp leaves its lanes' accumulator fragments (E
  // floats each, padded by 4 for conflict-free 16-byte access) in its own ring,
  // which is free once the warp's copies have landed
  static constexpr int kE = (D / 16) * NT * 4;
  static constexpr int kFragBytes = 32 * (kE + 4) * 4;
  // value scales of the group's KV head, staged with the query and read by the
  // epilogue, then the merge scalars: m and l of the warps x 16 heads
  static constexpr int kVsOffset = kLoopBytes;
  static constexpr int kScalOffset = kVsOffset + D * 4;
  static constexpr int kSmem = kScalOffset + 2 * kWarps * 16 * 4;
  static_assert(kFragBytes <= kWarpRing, "a warp's fragments fit its ring");
  static_assert(kChunks <= 32 && 32 % kChunks == 0, "row layout");
  static_assert(kCopies >= 1, "copy layout");
  static_assert(kGroups >= 1 && kThreads <= 1024, "CTA shape");
  // resident CTAs per SM the launch bounds promise (the register budget)
  static constexpr int kMinBlocks = SMALL ? kFitGroups : 1;
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// XOR swizzle of the 16-byte chunks of a dense shared-memory row, so that the
// 8 rows of an ldmatrix phase (and the rows a copy instruction writes) fall in
// distinct bank groups.
template <int ROW_BYTES>
__device__ __forceinline__ int swz(int r) {
  if constexpr (ROW_BYTES >= 128) {
    return r & 7;
  } else {
    return (r >> 1) & 3;  // 64-byte rows: two rows per 128-byte bank line
  }
}

// ---------------------------------------------------------------------------
// FP32 path of one CTA (onnxruntime PR 33707, Summary of Changes §1: a CTA
// that cannot bound the FP16 rounding evaluates its query heads in FP32 on the
// CUDA cores, starting from the inputs; review follow-up: value_scale folded
// into the numerator with a 2^80 shift for scores more than 80 nats below the
// maximum).  Same outputs as the tensor-core body for the CTA's (unit, split):
// O and lse with one split, else the partial (m, l, acc).  Two passes over the
// candidates (the maximum first, so nothing is rescaled), one warp per query
// head, lane l holding channels l, l + 32, ...  Slow by design: it runs only
// for CTAs that the eligibility checks send to it.
// ---------------------------------------------------------------------------
constexpr float kQueryErrorBudget = 0.125f;  // nats of logit shift from rounding Q' to fp16
constexpr float kTailDepth = 20.f;           // nats below the running maximum
constexpr float kMaxValueScale = 65536.f;    // |value_scale| above which the tail matters

template <int D, bool PAGED, bool FP16C, bool FP8, int kThreads>
__device__ __noinline__ void attend_fp32(const DecodeParams p, float* q32, const float* svs,
                                         int unit, int split, int chunk) {
  constexpr int kWarps = kThreads / 32;
  constexpr int C = D / 32;  // channels per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = p.G;
  // the CTA's range of positions [lo, hi) (the same rules as the tensor-core
  // body: the capacity, the clamped live length, the window start wlo and the
  // chunks counted from it rounded down to 16)
  const int row = unit / p.Hkv, g = unit - row * p.Hkv;
  const int cap = PAGED ? p.max_blocks * p.bs : p.max_sel;
  int len = cap, wlo = 0;
  if constexpr (PAGED) {
    len = min(max(p.seq_lens[row], 0), cap);
    if (p.window >= 0) wlo = max(0, len - 1 - p.window);
  }
  const int lo = (wlo & ~15) + split * chunk;
  const int hi = min(min(lo + chunk, cap), len);
  // Q * k_scale in fp32, not rounded to fp16
  const __half* qrow =
      reinterpret_cast<const __half*>(p.q) + ((long long)row * p.Hq + g * G) * D;
  for (int e = threadIdx.x; e < G * D; e += kThreads) {
    const int d = e % D;
    float x = __half2float(qrow[e]);
    if constexpr (!FP16C) x *= p.per_channel ? p.k_scale[g * D + d] : p.k_scale[0];
    q32[e] = x;
  }
  __syncthreads();
  // cache row of position t, or -1 if t is not attended
  auto row_of = [&](int t) -> long long {
    if constexpr (PAGED) {
      if (t < wlo) return -1;
      const int blk = p.block_table[(long long)row * p.max_blocks + t / p.bs];
      if (blk < 0 || (long long)blk >= p.cache_rows) return -1;
      return (long long)blk * p.bs + t % p.bs;
    } else {
      const int key = p.idx[(long long)row * p.max_sel + t];
      return key >= 0 && (long long)key < p.cache_rows ? key : -1;
    }
  };
  auto value = [&](const void* base, long long r, int d) -> float {
    const long long i = (r * p.Hkv + g) * D + d;
    if constexpr (FP16C) {
      return __half2float(reinterpret_cast<const __half*>(base)[i]);
    } else if constexpr (FP8) {
      const uint32_t code = reinterpret_cast<const uint8_t*>(base)[i];
      uint32_t lo2, hi2;
      e4m3x4_to_h2x2(code, lo2, hi2);
      return __half2float(__ushort_as_half(static_cast<unsigned short>(lo2 & 0xFFFFu)));
    } else {
      return static_cast<float>(reinterpret_cast<const int8_t*>(base)[i]);
    }
  };
  auto score = [&](const float* qh, long long r) -> float {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) acc = fmaf(qh[lane + 32 * c], value(p.k, r, lane + 32 * c), acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    float sc = acc * p.sigma;
    if constexpr (PAGED) {
      if (p.softcap > 0.f) sc = p.softcap * tanhf(sc / p.softcap);
    }
    return sc;
  };
  const bool direct = p.num_splits == 1;
  const long long head0 = (long long)row * p.Hq + g * G;
  for (int h = warp; h < G; h += kWarps) {
    const float* qh = q32 + h * D;
    float m = neg_inf();
    for (int t = lo; t < hi; ++t) {
      const long long r = row_of(t);
      if (r >= 0) m = fmaxf(m, score(qh, r));
    }
    // main accumulator (codes x weight) and the one for terms more than 80
    // nats down, kept 2^80 larger
    float l = 0.f, a[C], b[C];
#pragma unroll
    for (int c = 0; c < C; ++c) a[c] = b[c] = 0.f;
    if (m != neg_inf()) {
      for (int t = lo; t < hi; ++t) {
        const long long r = row_of(t);
        if (r < 0) continue;
        const float z = score(qh, r) - m;
        const float w = expf(z);
        l += w;
        if (z >= -80.f) {
#pragma unroll
          for (int c = 0; c < C; ++c) a[c] = fmaf(w, value(p.v, r, lane + 32 * c), a[c]);
        } else {
          const float ws = exp2f(fmaf(z, kLog2e, 80.f));
#pragma unroll
          for (int c = 0; c < C; ++c) b[c] = fmaf(ws, value(p.v, r, lane + 32 * c), b[c]);
        }
      }
    }
    if (direct) {
      float sc = 0.f;
      if (l > 0.f) {
        sc = 1.f / l;
        if (p.sink != nullptr) sc *= 1.f / (1.f + expf(p.sink[g * G + h] - (m + logf(l))));
      }
      __half* o = reinterpret_cast<__half*>(p.out) + (head0 + h) * D;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const int d = lane + 32 * c;
        const float vs = FP16C ? 1.f : svs[d];
        o[d] = __float2half_rn(sc == 0.f ? 0.f : (a[c] * vs + b[c] * (vs * 0x1p-80f)) * sc);
      }
      if (lane == 0 && p.lse != nullptr) p.lse[head0 + h] = l > 0.f ? m + logf(l) : neg_inf();
    } else {
      const long long base = ((long long)unit * p.num_splits + split) * G + h;
      if (l > 0.f) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
          const int d = lane + 32 * c;
          const float vs = FP16C ? 1.f : svs[d];
          p.ws_acc[base * D + d] = a[c] * vs + b[c] * (vs * 0x1p-80f);
        }
      }
      if (lane == 0) {
        p.ws_m[base] = l > 0.f ? m : neg_inf();
        p.ws_l[base] = l;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Longest-first dispatch (paged decode).  CTAs start in the order of their
// linear index, and a ragged batch otherwise leaves SMs idle at the end while
// the last long splits finish.  The CTA at dispatch position pos takes the
// item (unit, split) of rank pos in this order: the full chunks (split-major),
// then the partial chunks by size in quarters of a chunk (largest quarter
// first; row order within a quarter), then the empty ones (split-major).  A
// batch whose rows all have the same live length keeps the natural order,
// which is then already longest-first.  The geometry (num_splits, chunk) is
// untouched; only which CTA computes which split changes, so the results are
// the same bit for bit.
// Batches of up to 128 rows: lane l of every warp holds rows l, l + 32, ...,
// and each warp ranks on its own with ballots and shuffles (no shared memory,
// no barrier).
// The host enables it (DecodeParams::lpt) for chunks of at least 1280 tokens:
// a CTA whose item changes loads its prologue twice, which only long CTAs
// repay (measured on a ragged batch, kernel time against split-major order:
// -10 % with 2048-token chunks, -1 to -1.5 % with 1376 and 1648, +3 % with
// 1024, +4 to +8 % with 272 and 288).
// ---------------------------------------------------------------------------

// lane of the n-th (from 0) set bit of mask
__device__ __forceinline__ int nth_set_lane(unsigned mask, int n) {
  for (int i = 0; i < n; ++i) mask &= mask - 1u;
  return __ffs(mask) - 1;
}

static __device__ __noinline__ int2 lpt_item(const DecodeParams p, int pos) {
  constexpr int J = kLptMaxRows / 32;  // rows per lane: lane, lane + 32, ...
  const int lane = threadIdx.x & 31;
  const int B = p.rows, Hkv = p.Hkv, ns = p.num_splits, chunk = p.chunk;
  const int cap = p.max_blocks * p.bs;
  const int jn = (B + 31) / 32;  // row groups in use (uniform)
  // row lane + 32 j: nf full chunks, then a partial one of rem tokens (0: none)
  int nf[J], rem[J], eff[J];
  bool has[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int r = lane + 32 * j;
    has[j] = r < B;
    nf[j] = rem[j] = eff[j] = 0;
    if (has[j]) {
      const int live = min(max(p.seq_lens[r], 0), cap);
      const int base = p.window >= 0 ? (max(0, live - 1 - p.window) & ~15) : 0;
      eff[j] = live - base;
      nf[j] = min(ns, eff[j] / chunk);
      rem[j] = nf[j] < ns ? eff[j] - nf[j] * chunk : 0;
    }
  }
  // (every lane takes part in every shuffle and vote below: none sits inside a
  // condition that differs between lanes)
  const int eff0 = __shfl_sync(0xffffffffu, eff[0], 0);
  bool same = true;
#pragma unroll
  for (int j = 0; j < J; ++j) same &= !has[j] || eff[j] == eff0;
  if (__all_sync(0xffffffffu, same))
    return make_int2(blockIdx.x, blockIdx.y);  // uniform batch: already longest-first
  // the rank-th row (ascending) among those whose bit is set in m[j]
  auto nth_row = [&](const unsigned (&m)[J], int rank) -> int {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = __popc(m[j]);
      if (rank < c) return 32 * j + nth_set_lane(m[j], rank);
      rank -= c;
    }
    return -1;  // not reached
  };
  int cum = 0;
  for (int s = 0; s < ns; ++s) {  // full chunks, split-major
    unsigned m[J];
    int c = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      m[j] = j < jn ? __ballot_sync(0xffffffffu, has[j] && nf[j] > s) : 0u;
      c += __popc(m[j]);
    }
    if (pos < cum + Hkv * c) {
      const int q = pos - cum;
      return make_int2(nth_row(m, q / Hkv) * Hkv + q % Hkv, s);
    }
    cum += Hkv * c;
  }
  for (int qt = 3; qt >= 0; --qt) {  // partial chunks, largest quarter first
    unsigned m[J];
    int c = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      m[j] = j < jn ? __ballot_sync(0xffffffffu, has[j] && rem[j] > 0 &&
                                                     (4 * rem[j]) / chunk == qt)
                    : 0u;
      c += __popc(m[j]);
    }
    if (pos < cum + Hkv * c) {
      const int q = pos - cum;
      const int r = nth_row(m, q / Hkv);
      int nfr = 0;  // nf of row r, from the lane that holds it
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int v = __shfl_sync(0xffffffffu, nf[j], r & 31);
        if (j == r / 32) nfr = v;
      }
      return make_int2(r * Hkv + q % Hkv, nfr);
    }
    cum += Hkv * c;
  }
  for (int s = 0; s < ns; ++s) {  // empty chunks, split-major
    unsigned m[J];
    int c = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = nf[j] + (rem[j] > 0 ? 1 : 0);  // first empty split of the row
      m[j] = j < jn ? __ballot_sync(0xffffffffu, has[j] && e <= s) : 0u;
      c += __popc(m[j]);
    }
    if (pos < cum + Hkv * c) {
      const int q = pos - cum;
      return make_int2(nth_row(m, q / Hkv) * Hkv + q % Hkv, s);
    }
    cum += Hkv * c;
  }
  return make_int2(blockIdx.x, blockIdx.y);  // not reached: the ranks cover the grid
}

// ---------------------------------------------------------------------------
// Balanced pieces (paged, chunk 0 on the API).  The split geometry of the
// pages fixes a chunk from the capacity, so a ragged batch's longest rows
// carry chunks of the full length while the short rows' CTAs finish early.
// Here the grid and the partial slots still come from the capacity and the
// row count alone (capture-safe), but each CTA derives its piece on the device
// from all live lengths: row b gets n_b = min(S, 1 + floor(eff_b * (P - B) /
// sum eff)) pieces (S partial slots per row, P the (row, piece) pairs the
// batch may use, about one wave of CTAs over the KV heads), each
// ceil(eff_b / n_b) rounded up to the CTA's round of positions, and n_b
// recomputed from that.  The pieces are dealt piece-index-major: all rows'
// first pieces, then the second pieces of the rows that have one, ...  CTA c
// also marks the partial slots 2c and 2c + 1 (unit-major) empty when no piece
// uses them, so the combine sees (m = -inf, l = 0) there.
// Returns (unit, piece, piece length, 1), or (.., 0) for a CTA without a piece.
// ---------------------------------------------------------------------------
static __device__ __noinline__ int4 balanced_item(const DecodeParams p, int c) {
  constexpr int J = kLptMaxRows / 32;  // rows per lane: lane, lane + 32, ...
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = p.rows, Hkv = p.Hkv, S = p.num_splits, rnd = p.bal_round;
  const int cap = p.max_blocks * p.bs;
  const int jn = (B + 31) / 32;
  int eff[J], n[J], pl[J];
  bool has[J];
  long long tot = 0;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int r = lane + 32 * j;
    has[j] = r < B;
    eff[j] = 0;
    if (has[j]) {
      const int live = min(max(p.seq_lens[r], 0), cap);
      const int base = p.window >= 0 ? (max(0, live - 1 - p.window) & ~15) : 0;
      eff[j] = live - base;
    }
    tot += eff[j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const int extra = max(p.bal_pieces - B, 0);
#pragma unroll
  for (int j = 0; j < J; ++j) {
    int k = 1 + (tot > 0 ? (int)((long long)eff[j] * extra / tot) : 0);
    k = min(k, S);
    pl[j] = eff[j] > 0 ? (eff[j] + k - 1) / k : rnd;
    pl[j] = (pl[j] + rnd - 1) / rnd * rnd;
    n[j] = eff[j] > 0 ? (eff[j] + pl[j] - 1) / pl[j] : 1;
  }
  // value of row r's entry of a per-lane array (every lane takes part)
  auto of_row = [&](const int (&a)[J], int r) -> int {
    int out = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int v = __shfl_sync(0xffffffffu, a[j], r & 31);
      if (j == r / 32) out = v;
    }
    return out;
  };
  // the partial slots 2c, 2c + 1 that no piece fills: empty
  if (warp == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const long long t = 2LL * c + e;
      const int u = (int)(t / S), k = (int)(t - (long long)u * S);
      const int nu = u < B * Hkv ? of_row(n, u / Hkv) : 0;  // (uniform over the warp)
      if (u < B * Hkv && k >= nu && lane < p.G) {
        const long long sb = ((long long)u * S + k) * p.G + lane;
        p.ws_m[sb] = neg_inf();
        p.ws_l[sb] = 0.f;
      }
    }
  }
  // piece-index-major order: round k holds the rows with more than k pieces
  int cum = 0;
  for (int k = 0; k < S; ++k) {
    unsigned m[J];
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      m[j] = j < jn ? __ballot_sync(0xffffffffu, has[j] && n[j] > k) : 0u;
      cnt += __popc(m[j]);
    }
    if (cnt == 0) break;
    if (c < cum + Hkv * cnt) {
      const int q = c - cum;
      int rank = q / Hkv, r = -1;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int cj = __popc(m[j]);
        if (r < 0 && rank < cj) r = 32 * j + nth_set_lane(m[j], rank);
        if (r < 0) rank -= cj;
      }
      return make_int4(r * Hkv + q % Hkv, k, of_row(pl, r), 1);
    }
    cum += Hkv * cnt;
  }
  return make_int4(0, 0, 0, 0);
}

template <int D, int NT, bool PAGED, bool FP16C, bool PLO, bool FP8>
__global__ void __launch_bounds__((Tile<D, NT, FP16C, PAGED || !PLO>::kThreads),
                                  (Tile<D, NT, FP16C, PAGED || !PLO>::kMinBlocks))
decode_kernel(const DecodeParams p) {
  using T = Tile<D, NT, FP16C, PAGED || !PLO>;
  constexpr int kWarps = T::kWarps;
  constexpr int kThreads = T::kThreads;
  constexpr int KC = D / 16;  // k-chunks of QK^T and m-tiles of PV
  constexpr int SUB = T::SUB;
  extern __shared__ __align__(128) uint8_t smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int grp = lane >> 2;
  const int tig = lane & 3;
  const int G = p.G;
  const int cap = PAGED ? p.max_blocks * p.bs : p.max_sel;
  // block of a 16-aligned position and the row offset of that position in its
  // block (block_size is a multiple of 16; a shift when it is a power of two)
  const int bs_shift = p.bs_log2;
  auto block_of = [&](int pos) -> int { return bs_shift >= 0 ? pos >> bs_shift : pos / p.bs; };
  auto offset_in_block = [&](int pos) -> int {
    return bs_shift >= 0 ? pos & (p.bs - 1) : pos % p.bs;
  };
  grid_dependency_wait();  // inputs may come from the previous kernel of the stream

  // ---------------- the CTA's item (unit, split) and what depends on it ----------------
  // Loaded by `setup`: the query rows of the group and their key scales (8
  // channels per thread and step), the value scales of the KV head, the
  // length, the candidate range of the split and the first gather keys, all
  // issued together so that their latencies overlap.  A paged CTA then ranks
  // the batch for the longest-first dispatch (its loads overlap the ones
  // above) and loads again only if that gives it another item.
  constexpr int kQSteps = (NT * D + kThreads - 1) / kThreads;
  constexpr int kVsPer = (D + kThreads - 1) / kThreads;
  struct Item {
    int unit, split, row, g, len, wlo, base, lo, nhi;
    uint4 q_raw[kQSteps];
    float4 ks_raw[kQSteps][2];
    float vs_raw[kVsPer];
    int pf[T::kStages + 1];
  };
  // The gather key of step k of this warp in [lo_, end) of row row_ (-1 past
  // the end): the list entry of position (lane % kStep) of the step (sparse),
  // or the block id of 16-token tile (lane % SUB) of the step (paged; block_size
  // is a multiple of 16).  Warp w takes the steps w, w + kWarps, ...
  auto key_of = [&](int row_, int lo_, int end, int k) -> int {
    const int n = end > lo_ ? (end - lo_ + T::kStep - 1) / T::kStep : 0;
    const int nw = n > warp ? (n - warp + kWarps - 1) / kWarps : 0;
    if (k >= nw) return -1;
    const int pos0 = lo_ + T::kStep * (warp + kWarps * k);
    if constexpr (PAGED) {
      const int pos = pos0 + kSub * (lane % SUB);
      return pos < end ? __ldg(p.block_table + (long long)row_ * p.max_blocks + block_of(pos)) : -1;
    } else {
      const int pos = pos0 + (lane % T::kStep);
      return pos < end ? __ldg(p.idx + (long long)row_ * p.max_sel + pos) : -1;
    }
  };
  auto setup = [&](int unit_, int split_, int chunk_, Item& it) {
    it.unit = unit_;
    it.split = split_;
    it.row = unit_ / p.Hkv;
    it.g = unit_ - it.row * p.Hkv;
    const __half* qrow =
        reinterpret_cast<const __half*>(p.q) + ((long long)it.row * p.Hq + it.g * G) * D;
#pragma unroll
    for (int i = 0; i < kQSteps; ++i) {
      const int e = threadIdx.x + i * kThreads;
      const int h = (e * 8) / D, d0 = (e * 8) % D;
      it.q_raw[i] = make_uint4(0u, 0u, 0u, 0u);
      it.ks_raw[i][0] = it.ks_raw[i][1] = make_float4(1.f, 1.f, 1.f, 1.f);
      if (e < NT * D && h < G) {
        it.q_raw[i] = *reinterpret_cast<const uint4*>(qrow + h * D + d0);
        if constexpr (!FP16C) {
          if (p.per_channel) {
            it.ks_raw[i][0] = *reinterpret_cast<const float4*>(p.k_scale + it.g * D + d0);
            it.ks_raw[i][1] = *reinterpret_cast<const float4*>(p.k_scale + it.g * D + d0 + 4);
          } else {
            const float k0 = p.k_scale[0];
            it.ks_raw[i][0] = it.ks_raw[i][1] = make_float4(k0, k0, k0, k0);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kVsPer; ++i) {
      const int d = threadIdx.x + i * kThreads;
      it.vs_raw[i] = 1.f;
      if constexpr (!FP16C) {
        if (d < D) it.vs_raw[i] = p.per_channel ? p.v_scale[it.g * D + d] : p.v_scale[0];
      }
    }
    // candidate range (positions fit 32 bits: the host checks cap + num_splits
    // * chunk <= INT32_MAX).  Sliding window (paged only): the query at
    // position len - 1 attends [wlo, len) with wlo = len - 1 - window; the
    // splits count their chunks from wlo rounded down to the 16-token tile
    // granule, so this one case waits for the length before the gather keys.
    it.len = 0;
    if constexpr (PAGED) it.len = p.seq_lens[it.row];  // in flight while the keys are fetched
    it.wlo = 0;
    it.base = 0;
    if constexpr (PAGED) {
      if (p.window >= 0) {
        const int live = min(max(it.len, 0), cap);
        it.wlo = max(0, live - 1 - p.window);
        it.base = it.wlo & ~15;
      }
    }
    it.lo = it.base + split_ * chunk_;
    it.nhi = min(it.lo + chunk_, cap);  // nominal end (capacity-bounded)
    // the first keys, fetched against the nominal end before the live length
    // of a paged sequence is known
#pragma unroll
    for (int k = 0; k <= T::kStages; ++k) it.pf[k] = key_of(it.row, it.lo, it.nhi, k);
  };
  Item it;
  int chunk = p.chunk;  // the CTA's piece length (balanced pieces: its own)
  if (PAGED && p.balanced) {
    const int4 x = balanced_item(p, blockIdx.y * gridDim.x + blockIdx.x);
    if (!x.w) return;  // no piece for this CTA (uniform: every warp computes the same)
    chunk = x.z;
    setup(x.x, x.y, chunk, it);
  } else {
    // one call site: the natural item, then (paged, rarely) the dispatched one
    int u = blockIdx.x, sp = blockIdx.y;
#pragma unroll 1
    for (int pass = 0;; ++pass) {
      setup(u, sp, chunk, it);
      if constexpr (!PAGED) {
        break;
      } else {
        if (!p.lpt || pass > 0) break;
        const int2 x = lpt_item(p, blockIdx.y * gridDim.x + blockIdx.x);
        if (x.x == u && x.y == sp) break;  // uniform over the CTA
        u = x.x;
        sp = x.y;
      }
    }
  }
  const int unit = it.unit, split = it.split, row = it.row, g = it.g;
  int len = it.len;
  const int wlo = it.wlo, lo = it.lo, nhi = it.nhi;
  uint4(&q_raw)[kQSteps] = it.q_raw;
  float4(&ks_raw)[kQSteps][2] = it.ks_raw;
  int(&pf)[T::kStages + 1] = it.pf;

  // value scales of this KV head, staged in shared memory for the epilogue
  float* svs = reinterpret_cast<float*>(smem + T::kVsOffset);
  bool vs_bad = false;  // a value scale is not finite
  if constexpr (!FP16C) {
#pragma unroll
    for (int i = 0; i < kVsPer; ++i) {
      const int d = threadIdx.x + i * kThreads;
      if (d < D) {
        svs[d] = it.vs_raw[i];
        vs_bad |= !(fabsf(it.vs_raw[i]) <= 3.4028235e38f);
      }
    }
  }
  constexpr int MT_ITERS = (KC + kWarps - 1) / kWarps;

  // ---------------- per-warp gather pipeline ----------------
  // Warp w takes the steps w, w + kWarps, ... of kStep consecutive positions.
  int* wmask = reinterpret_cast<int*>(smem + T::kRingBytes) + warp * 4;
  const uint32_t ring_addr = smem_addr(smem + warp * T::kWarpRing);

  const char* kbase = reinterpret_cast<const char*>(p.k);
  const char* vbase = reinterpret_cast<const char*>(p.v);
  const long long row_stride = (long long)p.Hkv * T::kRowBytes;  // bytes between tokens
  const int chunk_id = lane % T::kChunks;
  const int row_in_copy = lane / T::kChunks;
  const long long lane_off = (long long)g * T::kRowBytes + chunk_id * 16;

  auto step_pos = [&](int k) -> int { return lo + T::kStep * (warp + kWarps * k); };
  auto steps_below = [&](int end) -> int {
    const int n = end > lo ? (end - lo + T::kStep - 1) / T::kStep : 0;
    return n > warp ? (n - warp + kWarps - 1) / kWarps : 0;
  };
  // later keys: against the live end once it is known
  int fetch_hi = nhi;
  int fetch_n = steps_below(nhi);
  auto fetch = [&](int k) -> int {
    if (k >= fetch_n) return -1;
    return key_of(row, lo, fetch_hi, k);
  };

  // live end of the split
  int hi = nhi;
  if constexpr (PAGED) {
    if (len > cap || len < 0) {
      if (g == 0 && split == 0 && threadIdx.x == 0) flag_or(p.flags, I8KV_FLAG_LEN_CLAMPED);
      len = len < 0 ? 0 : cap;
    }
    hi = min(nhi, len);
    // debug output: the gathered row of every attended position of the row,
    // -1 elsewhere; the row's CTAs of KV head 0 interleave over [0, cap)
    if (p.slots_out != nullptr && g == 0) {
      for (int t = split * kThreads + threadIdx.x; t < cap; t += p.num_splits * kThreads) {
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
  const int my_n = steps_below(hi);
  fetch_hi = hi;
  fetch_n = my_n;

  auto issue = [&](int k, int key) {
    if (k < my_n) {
      const int pos0 = step_pos(k);
      const int st = k % T::kStages;
      const uint32_t dK = ring_addr + st * T::kStageBytes;
      const uint32_t dV = dK + T::kTileBytes;
      unsigned mask;
      if constexpr (PAGED) {
        const int nvalid = min(hi - pos0, T::kStep);
        mask = nvalid >= 32 ? 0xFFFFFFFFu : ((1u << nvalid) - 1u);
        // positions before the window start (first step of split 0 only)
        const int nbelow = wlo - pos0;
        if (nbelow > 0) mask &= nbelow >= 32 ? 0u : ~((1u << nbelow) - 1u);
        bool bad_blk = false;
#pragma unroll
        for (int s = 0; s < SUB; ++s) {
          const int blk = __shfl_sync(0xffffffffu, key, s);
          if (blk < 0 || (long long)blk >= p.cache_rows) {
            if (((mask >> (kSub * s)) & 0xFFFFu) != 0u) bad_blk = true;
            mask &= ~(0xFFFFu << (kSub * s));
          }
        }
        if (bad_blk && lane == 0) flag_or(p.flags, I8KV_FLAG_BAD_BLOCK);
        // first cache row of each 16-token tile: block * block_size + offset
        long long tile_row[SUB];
#pragma unroll
        for (int s = 0; s < SUB; ++s)
          tile_row[s] = (long long)__shfl_sync(0xffffffffu, key, s) * p.bs +
                        offset_in_block(pos0 + kSub * s);
#pragma unroll
        for (int i = 0; i < T::kCopies; ++i) {
          const int r = row_in_copy + i * T::kRowsPerCopy;
          const bool ok = (mask >> r) & 1u;
          const long long off = ok ? (tile_row[r / kSub] + (r % kSub)) * row_stride + lane_off : 0;
          const uint32_t so = r * T::kRowBytes + ((chunk_id ^ swz<T::kRowBytes>(r)) << 4);
          cp_async16(dK + so, kbase + off, ok ? 16u : 0u);
          cp_async16(dV + so, vbase + off, ok ? 16u : 0u);
        }
      } else {
        const bool ok_mine = key >= 0 && (long long)key < p.cache_rows;
        mask = __ballot_sync(0xffffffffu, ok_mine);
        if constexpr (T::kStep == 16) mask &= 0xFFFFu;
#pragma unroll
        for (int i = 0; i < T::kCopies; ++i) {
          const int r = row_in_copy + i * T::kRowsPerCopy;
          const int t = __shfl_sync(0xffffffffu, key, r);
          const bool ok = (mask >> r) & 1u;
          const long long off = ok ? (long long)t * row_stride + lane_off : 0;
          const uint32_t so = r * T::kRowBytes + ((chunk_id ^ swz<T::kRowBytes>(r)) << 4);
          cp_async16(dK + so, kbase + off, ok ? 16u : 0u);
          cp_async16(dV + so, vbase + off, ok ? 16u : 0u);
        }
      }
      if (lane == 0) wmask[st] = (int)mask;
    }
    cp_async_commit();
  };

  // Start the gathers first: the query staging below overlaps their latency.
#pragma unroll
  for (int k = 0; k < T::kStages - 1; ++k) issue(k, pf[k]);
  int q0 = pf[T::kStages - 1], q1 = pf[T::kStages];

  // A CTA without candidates (an empty split) publishes the empty partial
  // (m = -inf, l = 0) or, with one split, O = 0 and lse = -inf.  The branch is
  // uniform over the CTA.
  if (npos == 0) {
    cp_async_wait_all();
    const long long head0 = (long long)row * p.Hq + g * G;
    for (int e = threadIdx.x; e < G * (p.num_splits == 1 ? D : 1); e += kThreads) {
      if (p.num_splits == 1) {
        const int h = e / D, d = e % D;
        reinterpret_cast<__half*>(p.out)[(head0 + h) * D + d] = __float2half_rn(0.f);
        if (d == 0 && p.lse != nullptr) p.lse[head0 + h] = neg_inf();
      } else {
        const long long base = ((long long)unit * p.num_splits + split) * G + e;
        p.ws_m[base] = neg_inf();
        p.ws_l[base] = 0.f;
      }
    }
    return;
  }

  // ---------------- Q' = fp16(Q * k_scale), staged through shared memory ----------------
  // The CTA takes the FP32 path when an element of Q * k_scale is not finite or
  // beyond the fp16 range, when for some head eps = sigma * |code|max *
  // sum_d |Q'_d - fp16(Q'_d)| (a bound on the logit shift from rounding Q')
  // exceeds the budget, or when a value scale is not finite.
  __half* sq = reinterpret_cast<__half*>(smem + T::kRingBytes + T::kMaskBytes);
  bool use_fp32 = false;
  bool vs_big_cta = false;
  {
    constexpr float kCodeMax = FP8 ? 448.f : 128.f;
    bool bad = false, over = false;
#pragma unroll
    for (int i = 0; i < kQSteps; ++i) {
      const int e = threadIdx.x + i * kThreads;
      if (e >= NT * D) break;  // uniform per warp (NT * D is a multiple of 32)
      const int h = (e * 8) / D, d0 = (e * 8) % D;
      uint4 packed = q_raw[i];
      if constexpr (!FP16C) {
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
        packed = make_uint4(w[0], w[1], w[2], w[3]);
        // sum over the D / 8 consecutive lanes holding this head's pieces
#pragma unroll
        for (int o = 1; o < D / 8 && o < 32; o <<= 1) err += __shfl_xor_sync(0xffffffffu, err, o);
        over |= h < G && p.sigma * kCodeMax * err > kQueryErrorBudget;
      }
      *reinterpret_cast<uint4*>(sq + h * T::kQStride + d0) = packed;
    }
    if (bad) flag_or(p.flags, I8KV_FLAG_QUERY_RANGE);
    use_fp32 = __syncthreads_or(bad || over || vs_bad);
    // some |value_scale| above 2^16 (the staged scales are visible after the
    // barrier; each warp reads them all, so no second barrier is needed)
    if constexpr (!FP16C) {
      bool big = false;
#pragma unroll
      for (int d = lane; d < D; d += 32) big |= fabsf(svs[d]) > kMaxValueScale;
      vs_big_cta = __any_sync(0xffffffffu, big);
    }
  }
  if (use_fp32) {
    cp_async_wait_all();
    __syncthreads();  // every warp's gathers have landed: the ring is free
    if (threadIdx.x == 0) flag_or(p.flags, I8KV_FLAG_FP32_PATH);
    attend_fp32<D, PAGED, FP16C, FP8, kThreads>(p, reinterpret_cast<float*>(smem), svs, unit,
                                                split, chunk);
    return;
  }
  // B fragments of Q'^T (k = channel, n = head) in the contraction order of the
  // K fragments: int8 caches take channels 16kc + 4tig + {0,1} / {2,3}, fp16
  // caches the natural 16kc + 2tig + {0,1} / {8,9}.
  uint32_t qf[NT][KC][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const __half* qh = sq + (nt * 8 + grp) * T::kQStride;
#pragma unroll
    for (int kc = 0; kc < KC; ++kc) {
      if constexpr (FP16C) {
        qf[nt][kc][0] = *reinterpret_cast<const uint32_t*>(qh + 16 * kc + 2 * tig);
        qf[nt][kc][1] = *reinterpret_cast<const uint32_t*>(qh + 16 * kc + 2 * tig + 8);
      } else {
        const uint2 v = *reinterpret_cast<const uint2*>(qh + 16 * kc + 4 * tig);
        qf[nt][kc][0] = v.x;
        qf[nt][kc][1] = v.y;
      }
    }
  }

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

  bool deep = false;

  // ldmatrix lane address: matrix m = lane/8 covers tokens (lane%8) + 8*(m&1)
  // of the tile and 16-byte chunk 2*c2 + (m>>1)
  const int ld_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int ld_sw = swz<T::kRowBytes>(ld_row);
  const int ld_hi = lane >> 4;
  const uint32_t ld_base = ld_row * T::kRowBytes;
  const float sigma = p.sigma;
  const float softcap = p.softcap;
  const float cap_k = 2.f * kLog2e / softcap;  // used only when softcap > 0

  // The main loop, instantiated twice: with the tail-depth tracking (a CTA with
  // some |value_scale| above 2^16) and without it (every other CTA), so that
  // the common loop carries none of it.
  auto main_loop = [&](auto track_tag) {
  constexpr bool kTrackDeep = decltype(track_tag)::value;
  for (int k = 0; k < my_n; ++k) {
    issue(k + T::kStages - 1, q0);
    q0 = q1;
    q1 = fetch(k + T::kStages + 1);
    cp_async_wait<T::kStages - 1>();
    __syncwarp();

    const int st = k % T::kStages;
    const uint32_t sK = ring_addr + st * T::kStageBytes;
    const uint32_t sV = sK + T::kTileBytes;
    const unsigned mask = (unsigned)wmask[st];

    // ---- S^T = K Q'^T per 16-token tile (with SUB = 1, two accumulator
    // chains over the k-chunks, summed after) ----
    float sacc[SUB][NT][4], sacc2[NT][4];
#pragma unroll
    for (int s = 0; s < SUB; ++s)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[s][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc2[nt][e] = 0.f;
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
      const uint32_t tK = sK + s * kSub * T::kRowBytes;
#pragma unroll
      for (int c2 = 0; c2 < T::kChunks / 2; ++c2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(tK + ld_base + (((2 * c2 + ld_hi) ^ ld_sw) << 4), r0, r1, r2, r3);
        if constexpr (FP16C) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (SUB == 1 && (c2 & 1))
              mma16816(sacc2[nt], r0, r1, r2, r3, qf[nt][c2][0], qf[nt][c2][1]);
            else
              mma16816(sacc[s][nt], r0, r1, r2, r3, qf[nt][c2][0], qf[nt][c2][1]);
          }
        } else {
          // K codes -> fp16 pairs (channel 4t, 4t+1) and (4t+2, 4t+3) of each
          // 4-byte word: the permuted contraction order of the Q' fragments
          uint32_t k0[4], k1[4];
          if constexpr (FP8) {
            e4m3x4_to_h2x2(r0, k0[0], k0[2]);
            e4m3x4_to_h2x2(r1, k0[1], k0[3]);
            e4m3x4_to_h2x2(r2, k1[0], k1[2]);
            e4m3x4_to_h2x2(r3, k1[1], k1[3]);
          } else {
            const uint32_t x0 = flip_i8x4(r0), x1 = flip_i8x4(r1);
            const uint32_t x2 = flip_i8x4(r2), x3 = flip_i8x4(r3);
            k0[0] = i8x2_to_h2(x0, 0x4140u);
            k0[1] = i8x2_to_h2(x1, 0x4140u);
            k0[2] = i8x2_to_h2(x0, 0x4342u);
            k0[3] = i8x2_to_h2(x1, 0x4342u);
            k1[0] = i8x2_to_h2(x2, 0x4140u);
            k1[1] = i8x2_to_h2(x3, 0x4140u);
            k1[2] = i8x2_to_h2(x2, 0x4342u);
            k1[3] = i8x2_to_h2(x3, 0x4342u);
          }
          {
            const uint32_t a0 = k0[0], a1 = k0[1], a2 = k0[2], a3 = k0[3];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816(sacc[s][nt], a0, a1, a2, a3, qf[nt][2 * c2][0], qf[nt][2 * c2][1]);
          }
          {
            const uint32_t a0 = k1[0], a1 = k1[1], a2 = k1[2], a3 = k1[3];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (SUB == 1)
                mma16816(sacc2[nt], a0, a1, a2, a3, qf[nt][2 * c2 + 1][0], qf[nt][2 * c2 + 1][1]);
              else
                mma16816(sacc[s][nt], a0, a1, a2, a3, qf[nt][2 * c2 + 1][0], qf[nt][2 * c2 + 1][1]);
            }
          }
        }
      }
    }
    if constexpr (SUB == 1) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[0][nt][e] += sacc2[nt][e];
    }

    // ---- online softmax (natural log domain) over the step's tokens ----
    uint32_t ph[SUB][NT][2], pl[SUB][NT][2];
    float alpha[NT][2];
    bool changed = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float sc[SUB][4];
#pragma unroll
      for (int s = 0; s < SUB; ++s)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[s][e] = sacc[s][nt][e] * sigma;
      if constexpr (PAGED) {
        if (softcap > 0.f) {
#pragma unroll
          for (int s = 0; s < SUB; ++s)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[s][e] = soft_cap(sc[s][e], softcap, cap_k);
        }
      }
#pragma unroll
      for (int s = 0; s < SUB; ++s) {
        const bool v_top = (mask >> (kSub * s + grp)) & 1u;
        const bool v_bot = (mask >> (kSub * s + grp + 8)) & 1u;
        if (!v_top) sc[s][0] = sc[s][1] = neg_inf();
        if (!v_bot) sc[s][2] = sc[s][3] = neg_inf();
      }
      float pr[SUB][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {  // head 2*tig + j of this n-tile
        float mx = fmaxf(sc[0][j], sc[0][2 + j]);
#pragma unroll
        for (int s = 1; s < SUB; ++s) mx = fmaxf(mx, fmaxf(sc[s][j], sc[s][2 + j]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(mrun[nt][j], mx);
        const float base = mnew == neg_inf() ? 0.f : mnew;
        if constexpr (kTrackDeep) {  // a valid score more than kTailDepth below the running max
#pragma unroll
          for (int s = 0; s < SUB; ++s)
            deep |= (sc[s][j] != neg_inf() && sc[s][j] < mnew - kTailDepth) ||
                    (sc[s][2 + j] != neg_inf() && sc[s][2 + j] < mnew - kTailDepth);
        }
        changed |= mnew != mrun[nt][j];
        alpha[nt][j] = fast_exp2((mrun[nt][j] - base) * kLog2e);
        float lsum = 0.f;
#pragma unroll
        for (int s = 0; s < SUB; ++s) {
          pr[s][j] = fast_exp2((sc[s][j] - base) * kLog2e);
          pr[s][2 + j] = fast_exp2((sc[s][2 + j] - base) * kLog2e);
          lsum += pr[s][j] + pr[s][2 + j];
        }
        lrun[nt][j] = lrun[nt][j] * alpha[nt][j] + lsum;
        mrun[nt][j] = mnew;
      }
      // probability tile p * 2^15 (high part, and for decode the residual)
#pragma unroll
      for (int s = 0; s < SUB; ++s) {
        __half hh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) hh[e] = __float2half_rn(pr[s][e] * kProbScale);
        ph[s][nt][0] = movm_t(pack_h2(hh[0], hh[1]));
        ph[s][nt][1] = movm_t(pack_h2(hh[2], hh[3]));
        if constexpr (PLO) {
          __half hl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            hl[e] = __float2half_rn(pr[s][e] * kProbScale - __half2float(hh[e]));
          pl[s][nt][0] = movm_t(pack_h2(hl[0], hl[1]));
          pl[s][nt][1] = movm_t(pack_h2(hl[2], hl[3]));
        }
      }
    }
    // rescale the accumulators only when some running maximum moved
    if (__any_sync(0xffffffffu, changed)) {
#pragma unroll
      for (int mt = 0; mt < KC; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[mt][nt][0] *= alpha[nt][0];
          acc[mt][nt][2] *= alpha[nt][0];
          acc[mt][nt][1] *= alpha[nt][1];
          acc[mt][nt][3] *= alpha[nt][1];
        }
    }

    // ---- O^T += V^T P^T, one 16-token tile at a time ----
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
      const uint32_t tV = sV + s * kSub * T::kRowBytes;
#pragma unroll
      for (int c2 = 0; c2 < T::kChunks / 2; ++c2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(tV + ld_base + (((2 * c2 + ld_hi) ^ ld_sw) << 4), r0, r1, r2, r3);
        if constexpr (FP16C) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(acc[c2][nt], r0, r2, r1, r3, ph[s][nt][0], ph[s][nt][1]);
            if constexpr (PLO) mma16816(acc[c2][nt], r0, r2, r1, r3, pl[s][nt][0], pl[s][nt][1]);
          }
        } else {
          // V^T codes (from the transposing load) -> fp16 pairs of bytes
          // (0, 2) and (1, 3) of each word
          uint32_t v0[4], v1[4];
          if constexpr (FP8) {
            e4m3x4_to_h2x2(prmt(r0, 0u, 0x3120u), v0[0], v0[1]);
            e4m3x4_to_h2x2(prmt(r1, 0u, 0x3120u), v0[2], v0[3]);
            e4m3x4_to_h2x2(prmt(r2, 0u, 0x3120u), v1[0], v1[1]);
            e4m3x4_to_h2x2(prmt(r3, 0u, 0x3120u), v1[2], v1[3]);
          } else {
            const uint32_t x0 = flip_i8x4(r0), x1 = flip_i8x4(r1);
            const uint32_t x2 = flip_i8x4(r2), x3 = flip_i8x4(r3);
            v0[0] = i8x2_to_h2(x0, 0x4240u);
            v0[1] = i8x2_to_h2(x0, 0x4341u);
            v0[2] = i8x2_to_h2(x1, 0x4240u);
            v0[3] = i8x2_to_h2(x1, 0x4341u);
            v1[0] = i8x2_to_h2(x2, 0x4240u);
            v1[1] = i8x2_to_h2(x2, 0x4341u);
            v1[2] = i8x2_to_h2(x3, 0x4240u);
            v1[3] = i8x2_to_h2(x3, 0x4341u);
          }
          {
            const uint32_t a0 = v0[0], a1 = v0[1], a2 = v0[2], a3 = v0[3];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma16816(acc[2 * c2][nt], a0, a1, a2, a3, ph[s][nt][0], ph[s][nt][1]);
              if constexpr (PLO)
                mma16816(acc[2 * c2][nt], a0, a1, a2, a3, pl[s][nt][0], pl[s][nt][1]);
            }
          }
          {
            const uint32_t a0 = v1[0], a1 = v1[1], a2 = v1[2], a3 = v1[3];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma16816(acc[2 * c2 + 1][nt], a0, a1, a2, a3, ph[s][nt][0], ph[s][nt][1]);
              if constexpr (PLO)
                mma16816(acc[2 * c2 + 1][nt], a0, a1, a2, a3, pl[s][nt][0], pl[s][nt][1]);
            }
          }
        }
      }
    }
    __syncwarp();
  }
  };
  if (vs_big_cta)
    main_loop(std::true_type{});
  else
    main_loop(std::false_type{});
  cp_async_wait_all();

  // a large value scale with a deep candidate: some probability was below the
  // fp16 tile's range, so the CTA starts over on the FP32 path
  if (vs_big_cta && __syncthreads_or(deep)) {
    if (threadIdx.x == 0) flag_or(p.flags, I8KV_FLAG_FP32_PATH);
    attend_fp32<D, PAGED, FP16C, FP8, kThreads>(p, reinterpret_cast<float*>(smem), svs, unit,
                                                split, chunk);
    return;
  }

  // ---------------- merge the warps' partials ----------------
  // Each warp publishes its (m, l) per head (l first summed over the 8 lanes
  // that share a head pair) and its fragments as soon as its loop is done,
  // without waiting for the others; one barrier then makes them all visible.
  float* mw = reinterpret_cast<float*>(smem + T::kScalOffset);  // [warps][16]
  float* lw = mw + kWarps * 16;                                 // [warps][16]
  float lsum[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = lrun[nt][j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      lsum[nt][j] = l;
    }
  if (grp == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        mw[warp * 16 + nt * 8 + 2 * tig + j] = mrun[nt][j];
        lw[warp * 16 + nt * 8 + 2 * tig + j] = lsum[nt][j];
      }
  }
  // each lane's fragment in its warp's ring: [lane][E (+4 pad)]
  auto frag_of = [&](int w) -> float* {
    return reinterpret_cast<float*>(smem + w * T::kWarpRing);
  };
  {
    // a lane's fragment of n-tile nt holds heads nt*8 + 2tig (+1): lanes whose
    // heads are all padding (G not a multiple of 8) neither write nor read it
    float4* mine = reinterpret_cast<float4*>(frag_of(warp) + lane * (T::kE + 4));
#pragma unroll
    for (int mt = 0; mt < KC; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        if (nt * 8 + 2 * tig < G)
          mine[mt * NT + nt] = make_float4(acc[mt][nt][0], acc[mt][nt][1], acc[mt][nt][2],
                                           acc[mt][nt][3]);
  }
  __syncthreads();

  // Warp w finishes m-tiles w, w + kWarps, ... of the fragment of its lane
  // index.  Each thread forms the merge weights f_w = exp(m_w - M) of its own
  // heads (2 tig, 2 tig + 1 of each n-tile), with M and L, from the published
  // scalars: no second barrier.
  float fw[NT][2][kWarps], Mh[NT][2], Lh[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = nt * 8 + 2 * tig + j;
      float M = neg_inf();
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * 16 + h]);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = M == neg_inf() ? 0.f : fast_exp2((mw[w * 16 + h] - M) * kLog2e);
        fw[nt][j][w] = f;
        L += f * lw[w * 16 + h];
      }
      Mh[nt][j] = M;
      Lh[nt][j] = L;
    }

  const bool direct = p.num_splits == 1;
  const long long head0 = (long long)row * p.Hq + g * G;
#pragma unroll
  for (int i = 0; i < MT_ITERS; ++i) {
    const int mt = warp + i * kWarps;
    if (mt >= KC) break;
    int da, db;  // the two channels of this thread in m-tile mt
    if constexpr (FP16C) {
      da = 16 * mt + grp;
      db = da + 8;
    } else {
      da = 16 * mt + 2 * grp;
      db = da + 1;
    }
    float vsa = 1.f, vsb = 1.f;
    if constexpr (!FP16C) {
      vsa = svs[da];
      vsb = svs[db];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (nt * 8 + 2 * tig >= G) continue;  // padding heads only
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float4 v = reinterpret_cast<const float4*>(
            frag_of(w) + lane * (T::kE + 4))[mt * NT + nt];
        const float f0 = fw[nt][0][w], f1 = fw[nt][1][w];
        a.x += f0 * v.x;  // (head 2tig,   channel da)
        a.y += f1 * v.y;  // (head 2tig+1, channel da)
        a.z += f0 * v.z;  // (head 2tig,   channel db)
        a.w += f1 * v.w;  // (head 2tig+1, channel db)
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = nt * 8 + 2 * tig + j;
        if (h >= G) continue;
        const float va = j == 0 ? a.x : a.y;
        const float vb = j == 0 ? a.z : a.w;
        const float M = Mh[nt][j], L = Lh[nt][j];
        if (direct) {
          float oa = 0.f, ob = 0.f;
          if (L > 0.f) {
            float sc = kInvProbScale / L;
            if (p.sink != nullptr) sc *= 1.f / (1.f + expf(p.sink[g * G + h] - (M + logf(L))));
            oa = va * sc * vsa;
            ob = vb * sc * vsb;
          }
          __half* o = reinterpret_cast<__half*>(p.out) + (head0 + h) * D;
          if constexpr (FP16C) {
            o[da] = __float2half_rn(oa);
            o[db] = __float2half_rn(ob);
          } else {
            *reinterpret_cast<__half2*>(o + da) = __floats2half2_rn(oa, ob);
          }
        } else if (L > 0.f) {
          const long long base = ((long long)unit * p.num_splits + split) * G + h;
          float* o = p.ws_acc + base * D;
          if constexpr (FP16C) {
            o[da] = (va * kInvProbScale) * vsa;
            o[db] = (vb * kInvProbScale) * vsb;
          } else {
            *reinterpret_cast<float2*>(o + da) =
                make_float2((va * kInvProbScale) * vsa, (vb * kInvProbScale) * vsb);
          }
        }
      }
    }
  }
  // per-head scalars: m and l of the split, or the lse of the row
  if (warp == 0 && grp == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = nt * 8 + 2 * tig + j;
        if (h >= G) continue;
        const float M = Mh[nt][j], L = Lh[nt][j];
        if (direct) {
          if (p.lse != nullptr) p.lse[head0 + h] = L > 0.f ? M + logf(L) : neg_inf();
        } else {
          const long long base = ((long long)unit * p.num_splits + split) * G + h;
          p.ws_m[base] = L > 0.f ? M : neg_inf();
          p.ws_l[base] = L;
        }
      }
  }
}

}  // namespace i8kv
