// Tensor-core (tcgen05) sparse-candidate prefill over an INT8 cache.
//
// What it computes (onnxruntime PR 33707 "INT8-KV DynamicSparseAttention",
// Summary of Changes §1: the multi-row prefill over gathered candidates, no
// splits, the probability tile as a single FP16 tile): for every query row r
// and query head h (KV head g = h / G),
//   O[r, h] = sum_t e^(s_t - m) v_scale * V[t, g] / sum_t e^(s_t - m),
//   s_t = sigma * dot(fp16(Q[r, h] * k_scale), K codes[t, g]),
// over the valid entries t of the row's candidate list, then lse and the sink.
//
// Design (GB300): a prefill's rows select large overlapping subsets of one
// cache (2048 of the first 6-8k tokens per row in the pages' workload), so the
// kernel does not gather per row.  A CTA takes a tile of 128 query vectors of
// one KV head (the (row, head) pairs r*G + j, consecutive, so a tile spans
// about 128 / G rows), holds a bitmask of each of its rows' candidates in
// shared memory, and streams the cache positions those rows select in blocks
// of 128 contiguous tokens:
//   S[128 x 128] = Q'[128 x D] K_block^T     tcgen05 kind::f16, M=128, N=128
//   softmax over the block with the row's mask (a position not in the row's
//   list gets probability 0), the probability tile p * 2^15 as fp16, written
//   back into tensor memory over the block's scores
//   O[128 x D] += P[128 x 128] V_block         tcgen05 kind::f16, M=128, N=D,
//                                            P from tensor memory
// So each cache block is converted int8 -> fp16 once per tile instead of once
// per row that selects it, and both products are real dense contractions with
// the accumulators in tensor memory.  The cost is the masked positions'
// products (at the pages' density of one in four, 3-4x the selected flops),
// which the tensor cores absorb.
// The exponentials take a base that follows the running maximum lazily: it
// moves only once the maximum has outgrown it by more than kLazy = 0.5 nats
// (p <= e^0.5 keeps p * 2^15 under the fp16 maximum), so O is rescaled on few
// blocks; O, the row sum and lse all use that base, so the result is the same.
//
// Warp roles (one CTA per SM), in two forms:
//   warps 0-7  softmax and epilogue; warps q and q + 4 own query vectors
//              32q .. 32q + 31 of the tile (tensor-memory lanes), warp q the
//              first 64 positions of a block and the first D/2 output channels,
//              warp q + 4 the others; the pair exchanges its block maxima (and
//              at the end its row sums) through shared memory.
//   converting form (544 threads; dsa_prefill without a workspace):
//   warps 8-15 converters: load the raw int8 K and V rows of a block into
//              registers (one block ahead), convert them exactly to fp16 (K as
//              the K-major B operand of QK^T, V as the MN-major B operand of
//              PV), signal the MMA thread.
//   warp 16    lane 0 issues the MMAs; the warp owns the tensor memory.
//   staged form (320 threads; dsa_prefill_ws): prefill_stage_kernel first
//              writes every block's fp16 K and V exactly as the converters
//              would lay them out in shared memory, and every row's bitmask
//              (its other CTAs, one per row), which the tiles copy in;
//   warp 8     lane 0 issues the MMAs; the warp owns the tensor memory;
//   warp 9     lane 0 brings each K or V block in with one bulk copy (the
//              mbarrier counts the bytes), K one block ahead of V.
// In the staged form a tile's blocks may also be split over several CTAs
// (where the tiles alone would leave SMs idle): each takes the blocks of its
// rank range and the candidates at their positions, and writes the partials
// that the split-combine kernel merges (PR 33707 §2's partial layout).
// (An MMA instruction costs the same up to N = 128 columns and about twice as
// much at N = 256, measured on this part: 128-token blocks keep QK^T at N=128
// instead of wasting half of every instruction at N = 64.)
// Hand-offs are mbarriers: every wait is bounded (about a second, or at once
// after another thread gave up); a CTA that gives up writes NaN for its
// outputs and raises I8KV_FLAG_WAIT_TIMEOUT instead of hanging.
//
// The numerical rules of the other kernels hold: a query vector whose Q' is
// out of the fp16 range or whose folding error exceeds the budget, a row whose
// list repeats an entry (the bitmask cannot count it), a non-finite value
// scale, or a value scale above 2^16 with a score more than 20 nats below the
// running maximum send the vector to an FP32 CUDA-core evaluation over its
// list (two passes, the 2^80-shifted accumulator for terms more than 80 nats
// down), whose result replaces the tensor-core one.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>

#include "../../include/int8kv.h"
#include "device.cuh"
#include "internal.h"
#include "tc.cuh"

namespace i8kv {
namespace pf {

constexpr int BM = 128;  // query vectors per tile (tensor-memory lanes)
constexpr int BN = 128;  // cache positions per block
constexpr int kSoftWarps = 8;   // two per tensor-memory lane quarter (column halves)
constexpr int kCvtWarps = 8;
constexpr int kCvtThreads = 32 * kCvtWarps;
// Warp roles of the two forms: the converting form reads the int8 cache and
// converts it in the kernel (8 converter warps, then the MMA warp); the staged
// form copies fp16 operand images that prefill_stage_kernel made (one loader
// warp after the MMA warp).
template <bool STAGED>
struct Roles {
  static constexpr int kMmaWarp = STAGED ? kSoftWarps : kSoftWarps + kCvtWarps;
  static constexpr int kLoadWarp = kSoftWarps + 1;  // staged form only
  static constexpr int kThreads = 32 * (STAGED ? kSoftWarps + 2 : kSoftWarps + kCvtWarps + 1);
};
constexpr float kQueryBudget = 0.125f;  // nats (the decode kernels' query-folding budget)
constexpr float kTail = 20.f;           // nats below the running maximum
constexpr float kLazy = 0.5f;           // nats the maximum may outgrow the base
constexpr float kBigVs = 65536.f;       // |value_scale| above which the tail matters

// barrier slots (8 bytes each) in the misc area
// (buffer b of a double-buffered pair: slot + b)
enum Bar { kKFull, kKFree, kVFull, kSFull0, kSFull1, kPFull, kPVDone, kDone, kNumBars };
// int slots after the barriers
enum Slot { kTmem, kAbort, kPMin, kPMax, kNumFp32, kVsBig, kVsBad, kNumSlots };

template <int D>
struct Layout {
  static constexpr int kQBytes = BM * D * 2;        // Q' (A of QK^T), fp16
  static constexpr int kKVBytes = BN * D * 2;       // one fp16 K or V block
  static constexpr int kQ = 0;
  static constexpr int kK16 = kQ + kQBytes;
  static constexpr int kV16 = kK16 + kKVBytes;
  static constexpr int kVs = kV16 + kKVBytes;       // the KV head's value scales
  static constexpr int kKs = kVs + D * 4;           // and its key scales
  static constexpr int kMisc = kKs + D * 4;         // barriers, ints, the FP32 vector list
  static constexpr int kBarBytes = 128;
  static constexpr int kSlotOff = kMisc + kBarBytes;
  static constexpr int kListOff = kSlotOff + 64;    // BM uint16 vector indices
  // [3][2 halves][BM] floats: block maxima (two block parities), row sums
  static constexpr int kXchg = kListOff + 2 * BM;
  static constexpr int kVFlag = kXchg + 6 * BM * 4; // per vector: bit 0 / 1 = FP32 path
  static constexpr int kVote = kVFlag + BM;         // [2][4 quarters][2 halves] ints
  static constexpr int kMask = kVote + 64;          // row bitmasks, block flags, row flags
  // Q' and K use the 128-byte swizzled K-major layout: slabs of 64 values
  // (128-byte rows, chunks XOR-permuted by row mod 8) over all rows of the
  // operand, one slab after the other along K
  static constexpr int kSlabQ = BM * 128;           // one 64-channel slab of Q'
  static constexpr int kSlabK = BN * 128;           // one 64-channel slab of a K block
  // V (the MN-major B of PV) uses plain core matrices (8 positions x 16
  // bytes): byte stride between 8-position groups
  static constexpr int kGroupD = (D / 8) * 128;
  // tensor memory: S0, S1 (BN fp32 columns each; P, fp16 pairs, is written
  // over the first BN / 2 columns of its block's S), then O (D columns)
  static constexpr int kOCol = 2 * BN;
  static constexpr int kTmemCols = (kOCol + D) <= 256 ? 256 : 512;
  static_assert(kNumBars * 8 <= kBarBytes, "barriers");
  static_assert(kK16 % 1024 == 0, "swizzle atoms are 1024-byte aligned");
  static_assert(kMask % 16 == 0, "the row masks are copied in 16-byte pieces");
  static_assert(kNumSlots * 4 <= 64, "slots");
};

struct Args {
  DecodeParams p;
  const uint8_t* stage;  // staged form: the fp16 operand images (else null)
  // splits of each tile's blocks (1: the kernel writes O and lse; more: each
  // CTA writes the partials of its share, which the combine kernel merges)
  int nsplit;
  float* part_acc;     // [rows * Hkv, nsplit, G, D]   value-scaled accumulators
  float* part_m;       // [rows * Hkv, nsplit, G]      base of the exponentials
  float* part_l;       // [rows * Hkv, nsplit, G]      row sums
  // staged form: every row's candidate bitmask, made by prefill_stage_kernel
  uint32_t* gmask;     // [rows, mask_words]
  int* gdup;           // [rows]  1 where the row lists some position twice
  int tiles_per_head;  // ceil(rows * G / 128)
  int mask_rows;       // rows a tile can span
  int mask_words;      // ceil(N / 32), rounded up to a multiple of 4
  int nblocks;         // ceil(N / BN)
};

// Byte offset, inside a block's fp16 operand, of the 16-byte chunk c0
// (channels 8c0 .. 8c0 + 7) of position pr: K (swz) in the 128-byte swizzled
// K-major slabs, V in plain core matrices (8 positions x 16 bytes).
template <int D>
__device__ __forceinline__ uint32_t chunk_offset(int pr, int c0, bool swz) {
  using L = Layout<D>;
  return swz ? (c0 >> 3) * L::kSlabK + pr * 128 + (((c0 & 7) ^ (pr & 7)) << 4)
             : (pr >> 3) * L::kGroupD + (pr & 7) * 16 + c0 * 128;
}

// Exact int8 -> fp16 of 16 codes (one 16-byte chunk) in channel order.
__device__ __forceinline__ void cvt16(const uint4 raw, uint4& lo, uint4& hi) {
  const uint32_t x0 = flip_i8x4(raw.x), x1 = flip_i8x4(raw.y);
  const uint32_t x2 = flip_i8x4(raw.z), x3 = flip_i8x4(raw.w);
  lo = make_uint4(i8x2_to_h2(x0, 0x4140u), i8x2_to_h2(x0, 0x4342u), i8x2_to_h2(x1, 0x4140u),
                  i8x2_to_h2(x1, 0x4342u));
  hi = make_uint4(i8x2_to_h2(x2, 0x4140u), i8x2_to_h2(x2, 0x4342u), i8x2_to_h2(x3, 0x4140u),
                  i8x2_to_h2(x3, 0x4342u));
}

// The FP32 CUDA-core evaluation of one query vector over its row's list (one
// warp; lane l holds channels l, l + 32, ...).  Two passes: the maximum, then
// the weights; terms more than 80 nats down accumulate 2^80 larger.
template <int D>
__device__ __noinline__ void fp32_vector(const DecodeParams& p, int row, int h, int g,
                                         const float* svs, long long pos_lo, long long pos_hi,
                                         float* pacc, float* pm, float* pl) {
  constexpr int C = D / 32;
  const int lane = threadIdx.x & 31;
  const long long N = p.cache_rows;
  const __half* qv = reinterpret_cast<const __half*>(p.q) + ((long long)row * p.Hq + h) * D;
  float q32[C];
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int d = lane + 32 * c;
    q32[c] = __half2float(qv[d]) * (p.per_channel ? p.k_scale[g * D + d] : p.k_scale[0]);
  }
  const int32_t* list = p.idx + (long long)row * p.max_sel;
  const int8_t* kc = reinterpret_cast<const int8_t*>(p.k);
  const int8_t* vc = reinterpret_cast<const int8_t*>(p.v);
  auto score = [&](long long t) -> float {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c)
      acc = fmaf(q32[c], static_cast<float>(kc[(t * p.Hkv + g) * D + lane + 32 * c]), acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc * p.sigma;
  };
  // (a split covers the candidates at positions pos_lo .. pos_hi - 1)
  const long long lo = pos_lo > 0 ? pos_lo : 0, hi = pos_hi < N ? pos_hi : N;
  float m = neg_inf();
  for (int j = 0; j < p.max_sel; ++j) {
    const int t = list[j];
    if (t >= lo && t < hi) m = fmaxf(m, score(t));
  }
  float l = 0.f, a[C], b[C];
#pragma unroll
  for (int c = 0; c < C; ++c) a[c] = b[c] = 0.f;
  if (m != neg_inf()) {
    for (int j = 0; j < p.max_sel; ++j) {
      const int t = list[j];
      if (t < lo || t >= hi) continue;
      const float z = score(t) - m;
      const float w = expf(z);
      l += w;
      if (z >= -80.f) {
#pragma unroll
        for (int c = 0; c < C; ++c)
          a[c] = fmaf(w, static_cast<float>(vc[((long long)t * p.Hkv + g) * D + lane + 32 * c]),
                      a[c]);
      } else {
        const float ws = exp2f(fmaf(z, kLog2e, 80.f));
#pragma unroll
        for (int c = 0; c < C; ++c)
          b[c] = fmaf(ws, static_cast<float>(vc[((long long)t * p.Hkv + g) * D + lane + 32 * c]),
                      b[c]);
      }
    }
  }
  if (pm != nullptr) {
    // a split's partial: the value-scaled accumulator relative to e^m
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int d = lane + 32 * c;
      const float vs = svs[d];
      pacc[d] = l > 0.f ? a[c] * vs + b[c] * (vs * 0x1p-80f) : 0.f;
    }
    if (lane == 0) {
      *pm = l > 0.f ? m : neg_inf();
      *pl = l;
    }
    return;
  }
  float sc = 0.f;
  if (l > 0.f) {
    sc = 1.f / l;
    if (p.sink != nullptr) sc *= 1.f / (1.f + expf(p.sink[h] - (m + logf(l))));
  }
  __half* o = reinterpret_cast<__half*>(p.out) + ((long long)row * p.Hq + h) * D;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int d = lane + 32 * c;
    const float vs = svs[d];
    o[d] = __float2half_rn(sc == 0.f ? 0.f : (a[c] * vs + b[c] * (vs * 0x1p-80f)) * sc);
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[(long long)row * p.Hq + h] = l > 0.f ? m + logf(l) : neg_inf();
}

// The staged form's operand images, one per (KV head g, block b) in that
// order: the block's K exactly as the converters leave it in shared memory
// (fp16, 128-byte swizzled K-major slabs), then its V (plain core matrices);
// positions at or past N are zero.  One CTA per image; thread ct converts
// the same 32-byte pieces a converter thread would.
template <int D>
__global__ void __launch_bounds__(kCvtThreads) prefill_stage_kernel(const Args a, uint8_t* img) {
  using L = Layout<D>;
  const DecodeParams& p = a.p;
  constexpr int kPairs = BN * D / 32 / kCvtThreads;
  const int ct = threadIdx.x;
  grid_dependency_wait();  // the cache may come from the previous kernel of the stream
  if (blockIdx.x >= p.Hkv * a.nblocks) {
    // The CTAs after the images: row `row`'s candidate bitmask (in shared
    // memory, then written out whole) and whether the row lists some
    // position twice (its valid entries outnumber its mask bits).
    extern __shared__ uint32_t rmask[];  // mask_words, then two counters
    const int row = blockIdx.x - p.Hkv * a.nblocks;
    const int mw = a.mask_words, max_sel = p.max_sel;
    const long long N = p.cache_rows;
    uint32_t* cnt = rmask + mw;
    for (int w = ct; w < mw; w += kCvtThreads) rmask[w] = 0u;
    if (ct < 2) cnt[ct] = 0u;
    __syncthreads();
    const int32_t* list = p.idx + (long long)row * max_sel;
    // Thread ct takes kRun consecutive entries of each kRun * kCvtThreads:
    // neighbours in a sorted list share mask words, and the entries of a run
    // that fall in one word are ORed in with one shared-memory atomic.
    constexpr int kRun = 8;
    const bool vec4 = (max_sel & 3) == 0 && (reinterpret_cast<uintptr_t>(list) & 15) == 0;
    int nv = 0;
    for (int j0 = kRun * ct; j0 < max_sel; j0 += kRun * kCvtThreads) {
      int tv[kRun];
      if (vec4 && j0 + kRun <= max_sel) {
        const int4 x = __ldg(reinterpret_cast<const int4*>(list + j0));
        const int4 y = __ldg(reinterpret_cast<const int4*>(list + j0 + 4));
        tv[0] = x.x; tv[1] = x.y; tv[2] = x.z; tv[3] = x.w;
        tv[4] = y.x; tv[5] = y.y; tv[6] = y.z; tv[7] = y.w;
      } else {
#pragma unroll
        for (int u = 0; u < kRun; ++u) tv[u] = j0 + u < max_sel ? __ldg(list + j0 + u) : -1;
      }
      int cw = -1;
      uint32_t cb = 0u;
#pragma unroll
      for (int u = 0; u < kRun; ++u) {
        const int t = tv[u];
        if (t >= 0 && t < N) {
          if ((t >> 5) != cw) {
            if (cb != 0u) atomicOr(rmask + cw, cb);
            cw = t >> 5;
            cb = 0u;
          }
          cb |= 1u << (t & 31);
          ++nv;
        }
      }
      if (cb != 0u) atomicOr(rmask + cw, cb);
    }
    int nb = 0;
    __syncthreads();
    for (int w = ct; w < mw; w += kCvtThreads) {
      const uint32_t v = rmask[w];
      a.gmask[(long long)row * mw + w] = v;
      nb += __popc(v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      nv += __shfl_xor_sync(0xffffffffu, nv, o);
      nb += __shfl_xor_sync(0xffffffffu, nb, o);
    }
    if ((ct & 31) == 0) {
      atomicAdd(cnt, (uint32_t)nv);
      atomicAdd(cnt + 1, (uint32_t)nb);
    }
    __syncthreads();
    if (ct == 0) a.gdup[row] = cnt[1] < cnt[0] ? 1 : 0;
    return;
  }
  const int b = blockIdx.x % a.nblocks, g = blockIdx.x / a.nblocks;
  uint8_t* dst = img + ((long long)g * a.nblocks + b) * (2 * L::kKVBytes);
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const int8_t* src = reinterpret_cast<const int8_t*>(kv == 0 ? p.k : p.v);
    uint8_t* out = dst + kv * L::kKVBytes;
#pragma unroll
    for (int k = 0; k < kPairs; ++k) {
      const int q = ct + kCvtThreads * k;
      const int pr = q % BN, cp = q / BN;
      const long long pos = (long long)b * BN + pr;
      uint4 raw[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
      if (pos < p.cache_rows) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src + (pos * p.Hkv + g) * D + 32 * cp);
        raw[0] = __ldg(s4);
        raw[1] = __ldg(s4 + 1);
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint4 lo, hi;
        cvt16(raw[hh], lo, hi);
        const int c0 = 4 * cp + 2 * hh;
        *reinterpret_cast<uint4*>(out + chunk_offset<D>(pr, c0, kv == 0)) = lo;
        *reinterpret_cast<uint4*>(out + chunk_offset<D>(pr, c0 + 1, kv == 0)) = hi;
      }
    }
  }
}

template <int D, bool STAGED>
__global__ void __launch_bounds__(Roles<STAGED>::kThreads, 1) prefill_tc_kernel(const Args a) {
  using L = Layout<D>;
  constexpr int kThreads = Roles<STAGED>::kThreads;
  constexpr int kMmaWarp = Roles<STAGED>::kMmaWarp;
  const DecodeParams& p = a.p;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  auto bar = [&](int k) -> uint32_t { return sbase + L::kMisc + 8 * k; };
  volatile int* slot = reinterpret_cast<volatile int*>(smem + L::kSlotOff);
  int* slot_rw = reinterpret_cast<int*>(smem + L::kSlotOff);
  uint16_t* fplist = reinterpret_cast<uint16_t*>(smem + L::kListOff);
  float* svs = reinterpret_cast<float*>(smem + L::kVs);
  float* sks = reinterpret_cast<float*>(smem + L::kKs);
  uint32_t* mask = reinterpret_cast<uint32_t*>(smem + L::kMask);
  uint8_t* blk_any = reinterpret_cast<uint8_t*>(mask + a.mask_rows * a.mask_words);
  uint8_t* row_dup = blk_any + a.nblocks;

  // ---------------- the tile ----------------
  const int G = p.G, Hkv = p.Hkv;
  const long long N = p.cache_rows;
  // later rows (longer causal lists) first, the KV heads interleaved, so that
  // the CTAs start in about decreasing order of work across the whole grid
  // (the splits of a tile are consecutive CTAs)
  const int sidx = blockIdx.x % a.nsplit;
  const int tb = blockIdx.x / a.nsplit;
  const int g = tb % Hkv;
  const int t_in_head = a.tiles_per_head - 1 - tb / Hkv;
  const long long nvec = (long long)p.rows * G;
  const long long v0 = (long long)t_in_head * BM;
  // index of a query vector's partial of this split: unit row * Hkv + g (the
  // decode partials' layout, which the combine kernel reads)
  auto vpart = [&](int row, int h) -> long long {
    return (((long long)row * Hkv + g) * a.nsplit + sidx) * G + (h - g * G);
  };
  const int r_lo = (int)(v0 / G);
  const int r_hi = (int)((v0 + BM - 1 < nvec ? v0 + BM - 1 : nvec - 1) / G);
  const int nrows = r_hi - r_lo + 1;

  grid_dependency_wait();  // inputs may come from the previous kernel of the stream

  if (warp == kMmaWarp) {
    tc::tmem_alloc(sbase + L::kSlotOff + 4 * kTmem, L::kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar(kKFull), STAGED ? 1 : kCvtThreads);
    tc::mbar_init(bar(kKFree), 1);
    tc::mbar_init(bar(kVFull), STAGED ? 1 : kCvtThreads);
    tc::mbar_init(bar(kSFull0), 1);
    tc::mbar_init(bar(kSFull1), 1);
    tc::mbar_init(bar(kPFull), 32 * kSoftWarps);
    tc::mbar_init(bar(kPVDone), 1);
    tc::mbar_init(bar(kDone), 1);
    tc::fence_mbar_init();
    // the swizzled operand layouts need 1024-byte aligned buffers
    slot[kAbort] = (sbase & 1023u) != 0u;
    slot[kPMin] = INT_MAX;
    slot[kPMax] = -1;
    slot[kNumFp32] = 0;
    slot[kVsBig] = 0;
    slot[kVsBad] = 0;
  }
  for (int i = tid; i < nrows * a.mask_words; i += kThreads) mask[i] = 0u;
  for (int i = tid; i < a.nblocks; i += kThreads) blk_any[i] = 0;
  for (int i = tid; i < nrows; i += kThreads) row_dup[i] = 0;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = static_cast<uint32_t>(slot[kTmem]);

  // the query vector of each softmax-warp thread
  const int half = (warp >> 2) & 1;         // softmax warps: column half
  const int r = 32 * (warp & 3) + lane;      // softmax warps: the vector of this thread
  const long long vidx = v0 + r;
  const bool vec_live = warp < kSoftWarps && vidx < nvec;
  const int vrow = vec_live ? (int)(vidx / G) : r_lo;
  const int vh = vec_live ? g * G + (int)(vidx - (long long)vrow * G) : 0;
  const __half* qrow = reinterpret_cast<const __half*>(p.q) + ((long long)vrow * p.Hq + vh) * D;
  // raw query rows in the V buffer, 16-byte chunk c of row r at chunk
  // c ^ (r mod D/8) (conflict-free reads by the warps' consecutive rows)
  constexpr int kQChunks = D / 8;
  auto raw_q = [&](int c) -> uint32_t {
    return (uint32_t)(L::kV16 + r * D * 2 + 16 * (c ^ (r & (kQChunks - 1))));
  };

  // raw query rows into the V buffer (cp.async), first: they land while the
  // masks are made
  if (warp < kSoftWarps / 2 && vec_live) {
#pragma unroll 8
    for (int c = 0; c < kQChunks; ++c) cp_async16(sbase + raw_q(c), qrow + 8 * c, 16);
  }
  cp_async_commit();

  // ---------------- the rows' candidate bitmasks ----------------
  if constexpr (STAGED) {
    // prefill_stage_kernel made every row's bitmask (and its repeat flag):
    // the tile's rows' masks are consecutive in memory, one cp.async each
    // 16 bytes; then the blocks some row selects
    const int mw = a.mask_words;
    const uint32_t* gm = a.gmask + (long long)r_lo * mw;
    for (int k = tid; k < nrows * mw / 4; k += kThreads)
      cp_async16(sbase + L::kMask + 16 * k, gm + 4 * k, 16);
    cp_async_commit();
    for (int rr = tid; rr < nrows; rr += kThreads) row_dup[rr] = a.gdup[r_lo + rr] != 0 ? 1 : 0;
    cp_async_wait_all();
    __syncthreads();
    for (int b = tid; b < a.nblocks; b += kThreads) {
      uint32_t any = 0u;
      for (int rr = 0; rr < nrows; ++rr) {
        const uint4 v = *reinterpret_cast<const uint4*>(mask + rr * mw + (BN / 32) * b);
        any |= v.x | v.y | v.z | v.w;
      }
      blk_any[b] = any != 0u ? 1 : 0;
      if (any != 0u) {
        atomicMin(slot_rw + kPMin, b * BN);
        atomicMax(slot_rw + kPMax, b * BN);
      }
    }
  } else {
    // The tile's rows' lists are consecutive in memory: each thread takes
    // every kThreads-th group of four entries of them (one 16-byte load where
    // the lists' alignment allows, else one entry per group), kListBatch
    // groups in flight at a time (one dependent load per entry would wait out
    // a memory latency per kThreads entries).  A group's entries that fall in
    // one mask word are ORed in with one shared-memory atomic.
    constexpr int kListBatch = 8;
    const int32_t* lists = p.idx + (long long)r_lo * p.max_sel;
    const bool vec4 = (p.max_sel & 3) == 0 && (reinterpret_cast<uintptr_t>(lists) & 15) == 0;
    const int per = vec4 ? 4 : 1;  // entries per group
    int lo = INT_MAX, hi = -1;
    auto flush = [&](int rr, int w, uint32_t bits) {
      if (bits == 0u) return;
      if (atomicOr(mask + rr * a.mask_words + w, bits) & bits) row_dup[rr] = 1;  // repeated
      blk_any[w / (BN / 32)] = 1;
    };
    int rr = 0, j = tid * per;  // the row and list slot of this thread's next group
    while (rr < nrows && j >= p.max_sel) {
      j -= p.max_sel;
      ++rr;
    }
    while (rr < nrows) {
      int4 tv[kListBatch];
      int rv[kListBatch];
#pragma unroll
      for (int u = 0; u < kListBatch; ++u) {
        rv[u] = rr;
        tv[u] = make_int4(-1, -1, -1, -1);
        if (rr < nrows) {
          const int32_t* src = lists + (long long)rr * p.max_sel + j;
          if (vec4)
            tv[u] = __ldg(reinterpret_cast<const int4*>(src));
          else
            tv[u].x = __ldg(src);
        }
        j += kThreads * per;
        while (rr < nrows && j >= p.max_sel) {
          j -= p.max_sel;
          ++rr;
        }
      }
#pragma unroll
      for (int u = 0; u < kListBatch; ++u) {
        if (rv[u] >= nrows) continue;
        const int te[4] = {tv[u].x, tv[u].y, tv[u].z, tv[u].w};
        int cw = -1;
        uint32_t cb = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = te[e];
          if (t < 0 || t >= N) continue;
          const uint32_t bit = 1u << (t & 31);
          if ((t >> 5) != cw) {
            flush(rv[u], cw, cb);
            cw = t >> 5;
            cb = 0u;
          }
          if (cb & bit) row_dup[rv[u]] = 1;  // repeated within the group
          cb |= bit;
          lo = min(lo, t);
          hi = max(hi, t);
        }
        flush(rv[u], cw, cb);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0 && hi >= 0) {
      atomicMin(slot_rw + kPMin, lo);
      atomicMax(slot_rw + kPMax, hi);
    }
    cp_async_wait_all();  // the raw query rows
  }
  // value and key scales of the KV head
  for (int d = tid; d < D; d += kThreads) {
    const float vs = p.per_channel ? p.v_scale[g * D + d] : p.v_scale[0];
    sks[d] = p.per_channel ? p.k_scale[g * D + d] : p.k_scale[0];
    svs[d] = vs;
    if (!(fabsf(vs) <= 3.4028235e38f)) slot[kVsBad] = 1;
    if (fabsf(vs) > kBigVs) slot[kVsBig] = 1;
  }
  __syncthreads();
  const int pmax = slot[kPMax];
  const int tile_lo = pmax >= 0 ? slot[kPMin] / BN : 0;
  const int tile_hi = pmax >= 0 ? pmax / BN : -1;
  // Split sidx takes the tile's selected blocks of ranks [r0, r1), r0 =
  // sidx * cnt / nsplit, and the candidates at positions [pos_lo, pos_hi):
  // from its first block to the next split's first (split 0 from 0, the last
  // one to N), so that every candidate of the tile's rows falls in one split.
  int blo = tile_lo, bhi = tile_hi;
  long long pos_lo = 0, pos_hi = N;
  if (a.nsplit > 1) {
    int cnt = 0;
    for (int b = tile_lo; b <= tile_hi; ++b) cnt += blk_any[b];
    const int r0 = (int)((long long)sidx * cnt / a.nsplit);
    const int r1 = (int)((long long)(sidx + 1) * cnt / a.nsplit);
    int b0 = tile_hi + 1, b1 = tile_hi + 1, rank = 0;  // the blocks of ranks r0 and r1
    for (int b = tile_lo; b <= tile_hi; ++b) {
      if (!blk_any[b]) continue;
      if (rank == r0) b0 = b;
      if (rank == r1) b1 = b;
      ++rank;
    }
    blo = b0;
    bhi = b1 - 1;
    if (sidx > 0) pos_lo = (long long)b0 * BN;
    if (sidx < a.nsplit - 1) pos_hi = (long long)b1 * BN;
  }
  const bool vs_bad = slot[kVsBad] != 0;
  const bool vs_big = slot[kVsBig] != 0;
  // the blocks some row of the tile selects, in order: blo, next(blo), ...
  auto next_blk = [&](int b) -> int {
    ++b;
    while (b <= bhi && !blk_any[b]) ++b;
    return b;
  };
  const int first = (blo <= bhi && blk_any[blo]) ? blo : next_blk(blo);

  // ---------------- Q' = fp16(Q * k_scale) (softmax warps) ----------------
  // Threads (half, r) of the softmax warps stage half the channels of query
  // vector r (from the raw row in the V buffer) into row r of the A operand:
  // channels 8c..8c+7 go to slab c / 8, row r, chunk (c % 8) ^ (r % 8).
  uint8_t* vflag = smem + L::kVFlag;
  bool need_fp32 = false;
  if (warp < kSoftWarps) {
    uint8_t* qdst = smem + L::kQ + r * 128;
    bool bad = false;
    float err = 0.f;
    constexpr int kHalfChunks = kQChunks / 2;
    constexpr int kQBatch = kHalfChunks < 16 ? kHalfChunks : 16;
    for (int c0 = half * kHalfChunks; c0 < (half + 1) * kHalfChunks; c0 += kQBatch) {
      uint4 raw[kQBatch];
#pragma unroll
      for (int u = 0; u < kQBatch; ++u)
        raw[u] = vec_live ? *reinterpret_cast<const uint4*>(smem + raw_q(c0 + u))
                          : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < kQBatch; ++u) {
        const int c = c0 + u;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (vec_live) {
          const __half2* qh = reinterpret_cast<const __half2*>(&raw[u]);
          const float4 k0 = *reinterpret_cast<const float4*>(sks + 8 * c);
          const float4 k1 = *reinterpret_cast<const float4*>(sks + 8 * c + 4);
          const float ks[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(qh[e]);
            const float x0 = f.x * ks[2 * e], x1 = f.y * ks[2 * e + 1];
            bad |= !(fabsf(x0) <= 65504.f) || !(fabsf(x1) <= 65504.f);
            o[e] = pack_h2(x0, x1);
            const float2 rr2 = __half22float2(*reinterpret_cast<const __half2*>(&o[e]));
            err += fabsf(x0 - rr2.x) + fabsf(x1 - rr2.y);
          }
          w = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>(qdst + (c >> 3) * L::kSlabQ + (((c & 7) ^ (r & 7)) << 4)) = w;
      }
    }
    // the halves' folding-error sums and range flags meet in shared memory
    // (the pair of warps q, q + 4 on named barrier 1 + q)
    float* qx = reinterpret_cast<float*>(smem + L::kXchg);  // [2][BM] errors, [2][BM] flags
    qx[half * BM + r] = err;
    qx[(2 + half) * BM + r] = bad ? 1.f : 0.f;
    asm volatile("bar.sync %0, %1;\n" ::"r"(1 + (warp & 3)), "r"(64) : "memory");
    if (half == 0) {
      const float err_all = err + qx[BM + r];
      const bool bad_all = bad || qx[3 * BM + r] != 0.f;
      if (vec_live) {
        if (bad_all) flag_or(p.flags, I8KV_FLAG_QUERY_RANGE);
        need_fp32 = bad_all || p.sigma * 128.f * err_all > kQueryBudget || vs_bad ||
                    row_dup[vrow - r_lo];
      }
      vflag[r] = need_fp32 ? 1 : 0;
    }
    tc::fence_smem_to_async();  // Q' is read by the tensor core
  }
  // a tile with nothing for the tensor cores (no selected block, or every
  // value scale unusable) skips the pipeline
  const bool run_tc = first <= bhi && !vs_bad;
  // the lists and raw query rows were read from the buffers that the bulk
  // copies (async proxy) fill next
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp < kSoftWarps) need_fp32 = vflag[r] != 0;

  // ---------------- the pipeline ----------------
  if (run_tc) {
    if (!STAGED && warp >= kSoftWarps && warp < kSoftWarps + kCvtWarps) {
      // ---- converters ----
      // Thread ct owns 32-byte pieces (row pr, channels 32cp .. 32cp + 31) of
      // every block's K and V: q = ct + 128k -> pr = q % BN, cp = q / BN, so
      // the lanes of a warp take consecutive rows (conflict-free core-matrix
      // stores).  Its pieces of the next block are loaded into registers while
      // the tensor cores work on the current ones.
      const int ct = tid - 32 * kSoftWarps;
      constexpr int kPairs = BN * D / 32 / kCvtThreads;
      const int8_t* kc = reinterpret_cast<const int8_t*>(p.k);
      const int8_t* vc = reinterpret_cast<const int8_t*>(p.v);
      uint4 kr[kPairs][2], vr[kPairs][2];
      auto load = [&](const int8_t* base, int blk, uint4 (&dst)[kPairs][2]) {
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
          const int q = ct + kCvtThreads * k;
          const long long pos = (long long)blk * BN + q % BN;
          if (pos < N) {
            // one 32-byte sector per lane, not kept in L1 (each is read once)
            const int8_t* src = base + (pos * Hkv + g) * D + 32 * (q / BN);
            asm volatile(
                "ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                : "=r"(dst[k][0].x), "=r"(dst[k][0].y), "=r"(dst[k][0].z), "=r"(dst[k][0].w),
                  "=r"(dst[k][1].x), "=r"(dst[k][1].y), "=r"(dst[k][1].z), "=r"(dst[k][1].w)
                : "l"(src));
          } else {
            dst[k][0] = dst[k][1] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      };
      // swz: K (128-byte swizzled slabs); else V (plain core matrices)
      auto convert = [&](const uint4 (&src)[kPairs][2], uint32_t dst16, bool swz) {
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
          const int q = ct + kCvtThreads * k;
          const int pr = q % BN, cp = q / BN;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint4 lo, hi;
            cvt16(src[k][hh], lo, hi);
            // channels 32cp + 16hh .. +15: 16-byte chunks c0 = 4cp + 2hh and c0 + 1
            const int c0 = 4 * cp + 2 * hh;
            const uint32_t a0 = dst16 + chunk_offset<D>(pr, c0, swz);
            const uint32_t a1 = dst16 + chunk_offset<D>(pr, c0 + 1, swz);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(a0), "r"(lo.x),
                         "r"(lo.y), "r"(lo.z), "r"(lo.w)
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(a1), "r"(hi.x),
                         "r"(hi.y), "r"(hi.z), "r"(hi.w)
                         : "memory");
          }
        }
      };
      // K runs one block ahead of V: K(i + 1) is converted once QK(i) has
      // read the K buffer, then V(i) once PV(i - 1) has read the V buffer
      load(kc, first, kr);
      load(vc, first, vr);
      bool ok = tc::mbar_wait(bar(kKFree), 1, slot);  // (passes at once)
      if (ok) {
        convert(kr, sbase + L::kK16, true);
        tc::fence_smem_to_async();
        tc::mbar_arrive(bar(kKFull));
        const int second = next_blk(first);
        if (second <= bhi) load(kc, second, kr);
      }
      int i = 0;
      for (int blk = first; ok && blk <= bhi; ++i) {
        const int nxt = next_blk(blk);
        // K(i + 1) first: its buffer frees when QK(i) completes, which comes
        // before PV(i - 1) is even issued
        if (nxt <= bhi) {
          if (!(ok = tc::mbar_wait(bar(kKFree), i & 1, slot))) break;
          convert(kr, sbase + L::kK16, true);
          tc::fence_smem_to_async();
          tc::mbar_arrive(bar(kKFull));
          const int nn = next_blk(nxt);
          if (nn <= bhi) load(kc, nn, kr);
        }
        if (!(ok = tc::mbar_wait(bar(kPVDone), (i & 1) ^ 1, slot))) break;
        convert(vr, sbase + L::kV16, false);
        tc::fence_smem_to_async();
        tc::mbar_arrive(bar(kVFull));
        if (nxt <= bhi) load(vc, nxt, vr);
        blk = nxt;
      }
      if (!ok) slot[kAbort] = 1;
    } else if (STAGED && warp == Roles<STAGED>::kLoadWarp) {
      // ---- loader (one thread): the blocks' fp16 operand images, K running
      // one block ahead of V exactly as the converters do ----
      if (lane == 0) {
        constexpr uint32_t kImg = 2 * L::kKVBytes;
        const uint8_t* img = a.stage + (long long)g * a.nblocks * kImg;
        int nk = 0, nv = 0;  // copies issued
        auto copy_in = [&](int blk, bool is_v) {
          const int b = is_v ? kVFull : kKFull;
          ++(is_v ? nv : nk);
          tc::mbar_arrive_expect_tx(bar(b), L::kKVBytes);
          tc::bulk_g2s(sbase + (is_v ? L::kV16 : L::kK16),
                       img + (long long)blk * kImg + (is_v ? L::kKVBytes : 0), L::kKVBytes,
                       bar(b));
        };
        bool ok = true;
        copy_in(first, false);
        int i = 0;
        for (int blk = first; blk <= bhi; ++i) {
          const int nxt = next_blk(blk);
          if (nxt <= bhi) {
            if (!(ok = tc::mbar_wait(bar(kKFree), i & 1, slot))) break;
            copy_in(nxt, false);
          }
          if (!(ok = tc::mbar_wait(bar(kPVDone), (i & 1) ^ 1, slot))) break;
          copy_in(blk, true);
          blk = nxt;
        }
        if (!ok) slot[kAbort] = 1;
        // every copy issued has landed before the loader leaves: the MMA
        // thread waited for each one it used; after an abort this waits
        // (bounded) for the others.  Only this thread arrives on the two
        // barriers, so the last copy's phase is the latest one.
        if (nk > 0 && !tc::mbar_wait(bar(kKFull), (nk - 1) & 1)) slot[kAbort] = 1;
        if (nv > 0 && !tc::mbar_wait(bar(kVFull), (nv - 1) & 1)) slot[kAbort] = 1;
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ---- MMA issue (one thread) ----
      // order: QK(0), QK(1), PV(0), QK(2), PV(1), ...: the scores of block
      // i + 1 are computed while the softmax works on block i
      if (lane == 0) {
        constexpr uint32_t kIdQK = tc::idesc_f16(BM, BN, false, false);
        constexpr uint32_t kIdPV = tc::idesc_f16(BM, D, false, true);
        const uint32_t q_s = sbase + L::kQ, k_s = sbase + L::kK16, v_s = sbase + L::kV16;
        auto pv = [&](int j) -> bool {
          if (!tc::mbar_wait(bar(kPFull), j & 1, slot)) return false;
          if (!tc::mbar_wait(bar(kVFull), j & 1, slot)) return false;
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            // A = P (tensor memory: lane = vector, fp16 pairs along the
            // positions), B = V (MN-major: K = positions, N = channels)
            const uint64_t bd = tc::smem_desc(v_s + kk * 2 * L::kGroupD, L::kGroupD, 128);
            // positions 64h .. 64h + 63 of the block (h = kk / 4) sit in
            // columns 64h .. 64h + 31 of its S buffer
            tc::mma_f16_ts(tbase + L::kOCol,
                           tbase + (j & 1) * BN + 64 * (kk >> 2) + 8 * (kk & 3), bd, kIdPV,
                           j > 0 || kk > 0);
          }
          tc::mma_commit(bar(kPVDone));
          return true;
        };
        int i = 0;
        bool ok = true;
        for (int blk = first; blk <= bhi; blk = next_blk(blk), ++i) {
          // S(i) overwrites P(i - 2): PV(i - 2) must have read it
          ok = tc::mbar_wait(bar(kKFull), i & 1, slot) &&
               (i < 2 || tc::mbar_wait(bar(kPVDone), i & 1, slot));
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // A = Q' (K-major: M = vectors, K = channels), B = K (K-major:
            // N = positions, K = channels)
            const uint32_t koff = (kk & 3) * 32;  // K step inside a 64-channel slab
            const uint64_t ad = tc::smem_desc_sw128(q_s + (kk >> 2) * L::kSlabQ + koff, 1024);
            const uint64_t bd = tc::smem_desc_sw128(k_s + (kk >> 2) * L::kSlabK + koff, 1024);
            tc::mma_f16(tbase + (i & 1) * BN, ad, bd, kIdQK, kk > 0);
          }
          tc::mma_commit(bar(kSFull0 + (i & 1)));
          tc::mma_commit(bar(kKFree));
          if (i > 0 && !(ok = pv(i - 1))) break;
        }
        if (ok && i > 0) ok = pv(i - 1);
        if (!ok) slot[kAbort] = 1;
        // everything issued has completed before the tensor memory is released
        tc::mma_commit(bar(kDone));
        if (!tc::mbar_wait(bar(kDone), 0)) slot[kAbort] = 1;
      }
      __syncwarp();
    } else if (warp < kSoftWarps) {
      // ---- softmax (one query vector per thread and column half) ----
      const uint32_t t_lane = (uint32_t)(32 * (warp & 3)) << 16;
      const uint32_t* mrow = mask + (vrow - r_lo) * a.mask_words;
      const float sigma = p.sigma;
      float* xchg = reinterpret_cast<float*>(smem + L::kXchg);  // [3][2][BM]
      float m_run = neg_inf(), m_top = neg_inf(), l_half = 0.f;
      bool deep = false, loop_ok = true;
      // the warp's lanes take every decision together (tcgen05.ld / st are
      // warp-collective)
      auto wait_all = [&](int b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, tc::mbar_wait(bar(b), parity, slot));
      };
      // the two warps of a lane quarter (64 threads, named barrier 1 + q)
      auto pair_sync = [&]() {
        asm volatile("bar.sync %0, %1;\n" ::"r"(1 + (warp & 3)), "r"(64) : "memory");
      };
      // Both warps of the pair take the same branch after every wait (so that
      // neither reaches a pair barrier the other has left): each publishes
      // its warp-uniform result, and both continue only if both succeeded.
      volatile int* votes = reinterpret_cast<volatile int*>(smem + L::kVote);
      int nvote = 0;
      auto pair_all = [&](bool ok) -> bool {
        volatile int* v = votes + (nvote++ & 1) * 8 + (warp & 3) * 2;
        if (lane == 0) v[half] = ok ? 1 : 0;
        pair_sync();
        return v[0] != 0 && v[1] != 0;
      };
      // the row's selection of 32 positions starting at 32 * word
      auto sel_word = [&](int word) -> uint32_t {
        return vec_live && word < a.mask_words ? mrow[word] : 0u;
      };
      int i = 0;
      for (int blk = first; blk <= bhi; blk = next_blk(blk), ++i) {
        if (!pair_all(wait_all(kSFull0 + (i & 1), (i >> 1) & 1))) {
          loop_ok = false;
          break;
        }
        tc::fence_after_sync();
        // this half's 64 positions: score columns 64h .. 64h + 63 of the block
        const uint32_t s_col = tbase + t_lane + (i & 1) * BN + 64 * half;
        // the half's 64 scores, read once: selected ones scaled by sigma,
        // the others -inf; the maximum over the half, then over the block
        // (with the other half's)
        float sv[64];
        tc::tmem_ld32(s_col, *reinterpret_cast<float(*)[32]>(&sv[0]));
        tc::tmem_ld32(s_col + 32, *reinterpret_cast<float(*)[32]>(&sv[32]));
        tc::tmem_wait_ld();
        float mx = neg_inf();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t w = sel_word(BN / 32 * blk + 2 * half + c);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = ((w >> j) & 1u) ? sv[32 * c + j] * sigma : neg_inf();
            sv[32 * c + j] = x;
            mx = fmaxf(mx, x);
          }
        }
        float* xb = xchg + (i & 1) * 2 * BM;
        xb[half * BM + r] = mx;
        pair_sync();
        mx = fmaxf(mx, xb[(half ^ 1) * BM + r]);
        const float top = fmaxf(m_top, mx);  // the running maximum
        // the base of the exponentials moves to the running maximum only once
        // that has grown by more than kLazy nats (p <= e^kLazy keeps p * 2^15
        // within fp16), so that O is rescaled only on those blocks
        const float m_new = top > m_run + kLazy ? top : m_run;
        const float base = m_new == neg_inf() ? 0.f : m_new;
        const float alpha = fast_exp2((m_run - base) * kLog2e);
        // probabilities p * 2^15 as fp16 pairs, written over the half's
        // scores (columns 64h .. 64h + 31)
        float ps = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ph[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float x0 = sv[32 * c + 2 * j], x1 = sv[32 * c + 2 * j + 1];
            if (vs_big)
              deep |= (x0 != neg_inf() && x0 < top - kTail) ||
                      (x1 != neg_inf() && x1 < top - kTail);
            // p * 2^15: the factor enters as 15 in the exponent (exact)
            const float p0 = fast_exp2(fmaf(x0 - base, kLog2e, 15.f));
            const float p1 = fast_exp2(fmaf(x1 - base, kLog2e, 15.f));
            ps += p0 + p1;
            ph[j] = pack_h2(p0, p1);
          }
          tc::tmem_st16u(s_col + 16 * c, ph);
        }
        l_half = l_half * alpha + ps * kInvProbScale;
        const bool rescale = i > 0 && m_new != m_run;
        m_run = m_new;
        m_top = top;
        // O is current once the previous block's PV has completed; this half
        // rescales channels hD/2 .. hD/2 + D/2 - 1.  (The wait stays even
        // when no vector rescales: it also keeps every softmax warp's arrival
        // for this block from counting toward the previous one.)
        const bool any_rescale = __any_sync(0xffffffffu, rescale);
        if (!pair_all(i == 0 || wait_all(kPVDone, (i - 1) & 1))) {
          loop_ok = false;
          break;
        }
        tc::fence_after_sync();
        if (any_rescale) {
          const float f = rescale ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            float o[32];
            const uint32_t oc = tbase + t_lane + L::kOCol + half * (D / 2) + 32 * c;
            tc::tmem_ld32(oc, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tc::tmem_st32(oc, o);
          }
        }
        tc::tmem_wait_st();  // P (and O) written before the MMA is told
        tc::fence_before_sync();
        tc::mbar_arrive(bar(kPFull));
      }
      // ---- epilogue: O / l, the sink, lse ----
      const bool ok = pair_all(__all_sync(0xffffffffu, loop_ok && !slot[kAbort]) &&
                               (i == 0 || wait_all(kPVDone, (i - 1) & 1)));
      tc::fence_after_sync();
      // the row sum and the tail flag of both halves (the pair left the loop
      // at the same block: every exit above follows a pair vote)
      float* lx = xchg + 4 * BM;
      lx[half * BM + r] = l_half;
      if (deep) atomicOr(reinterpret_cast<unsigned int*>(vflag) + (r >> 2), 2u << (8 * (r & 3)));
      pair_sync();
      const float l_run = l_half + lx[(half ^ 1) * BM + r];
      need_fp32 = vec_live && vflag[r] != 0;
      const bool write = vec_live && !need_fp32;
      if (a.nsplit > 1) {
        // this split's partial: O * 2^-15 * value_scale, relative to e^m_run
        const long long pv = vpart(vrow, vh);
        float* pacc = a.part_acc + pv * D;
        if (ok && i > 0) {
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            float o[32];
            const int d0 = half * (D / 2) + 32 * c;
            tc::tmem_ld32(tbase + t_lane + L::kOCol + d0, o);
            tc::tmem_wait_ld();
            if (write) {
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int d = d0 + 4 * u;
                *reinterpret_cast<float4*>(pacc + d) =
                    make_float4(o[4 * u] * kInvProbScale * svs[d],
                                o[4 * u + 1] * kInvProbScale * svs[d + 1],
                                o[4 * u + 2] * kInvProbScale * svs[d + 2],
                                o[4 * u + 3] * kInvProbScale * svs[d + 3]);
              }
            }
          }
        }
        if (ok && write && half == 0) {
          a.part_m[pv] = l_run > 0.f ? m_run : neg_inf();
          a.part_l[pv] = l_run;
        }
        if (!ok) slot[kAbort] = 1;
        if (half == 1) need_fp32 = false;  // one entry per vector in the FP32 list
        tc::fence_before_sync();
      } else {
      float sc = 0.f;
      const float lse_v = l_run > 0.f ? m_run + logf(l_run) : neg_inf();
      if (l_run > 0.f) {
        sc = kInvProbScale / l_run;
        if (p.sink != nullptr) sc *= 1.f / (1.f + expf(p.sink[vh] - lse_v));
      }
      __half* orow = reinterpret_cast<__half*>(p.out) + ((long long)vrow * p.Hq + vh) * D;
      if (ok && i > 0) {
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          float o[32];
          const int d0 = half * (D / 2) + 32 * c;
          tc::tmem_ld32(tbase + t_lane + L::kOCol + d0, o);
          tc::tmem_wait_ld();
          if (write) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint32_t h[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int d = d0 + 8 * u + 2 * e;
                h[e] = pack_h2(o[8 * u + 2 * e] * sc * svs[d], o[8 * u + 2 * e + 1] * sc * svs[d + 1]);
              }
              *reinterpret_cast<uint4*>(orow + d0 + 8 * u) = make_uint4(h[0], h[1], h[2], h[3]);
            }
          }
        }
      } else if (ok && write) {  // no selected block: O = 0
        for (int c = 0; c < D / 16; ++c)
          *reinterpret_cast<uint4*>(orow + half * (D / 2) + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
      }
      if (ok && write && half == 0 && p.lse != nullptr) p.lse[(long long)vrow * p.Hq + vh] = lse_v;
      if (!ok) slot[kAbort] = 1;
      if (half == 1) need_fp32 = false;  // one entry per vector in the FP32 list
      tc::fence_before_sync();
      }
    }
  } else if (warp < kSoftWarps / 2 && vec_live && !need_fp32) {
    // no tensor-core work: every position of the tile (or of this split) is
    // unselected
    if (a.nsplit > 1) {
      const long long pv = vpart(vrow, vh);
      a.part_m[pv] = neg_inf();
      a.part_l[pv] = 0.f;
    } else {
      __half* orow = reinterpret_cast<__half*>(p.out) + ((long long)vrow * p.Hq + vh) * D;
      for (int c = 0; c < D / 8; ++c)
        *reinterpret_cast<uint4*>(orow + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
      if (p.lse != nullptr) p.lse[(long long)vrow * p.Hq + vh] = neg_inf();
    }
  }
  if (!run_tc && warp >= kSoftWarps / 2) need_fp32 = false;  // listed by the first half
  if (need_fp32) {
    const int k = atomicAdd(slot_rw + kNumFp32, 1);
    fplist[k] = (uint16_t)r;
  }
  __syncthreads();

  const bool aborted = slot[kAbort] != 0;
  if (aborted) {
    // the CTA gave up waiting: its outputs are marked invalid
    if (tid == 0) flag_or(p.flags, I8KV_FLAG_WAIT_TIMEOUT);
    if (warp < kSoftWarps / 2 && vec_live) {
      if (a.nsplit > 1) {
        // a partial the combine cannot select away: m = +inf makes the
        // merged weights, O and lse NaN
        const long long pv = vpart(vrow, vh);
        for (int d = 0; d < D; ++d) a.part_acc[pv * D + d] = __int_as_float(0x7FC00000);
        a.part_m[pv] = __int_as_float(0x7F800000);
        a.part_l[pv] = __int_as_float(0x7FC00000);
      } else {
        __half* orow = reinterpret_cast<__half*>(p.out) + ((long long)vrow * p.Hq + vh) * D;
        for (int d = 0; d < D; ++d) orow[d] = __ushort_as_half(0x7E00);
        if (p.lse != nullptr) p.lse[(long long)vrow * p.Hq + vh] = __int_as_float(0x7FC00000);
      }
    }
  } else {
    // ---------------- the FP32 vectors (every warp takes its share) ----------------
    const int nfp = slot[kNumFp32];
    if (nfp > 0 && tid == 0) flag_or(p.flags, I8KV_FLAG_FP32_PATH);
    for (int k = warp; k < nfp; k += kThreads / 32) {
      const long long v = v0 + fplist[k];
      const int row = (int)(v / G);
      const int h = g * G + (int)(v - (long long)row * G);
      if (a.nsplit > 1) {
        const long long pv = vpart(row, h);
        fp32_vector<D>(p, row, h, g, svs, pos_lo, pos_hi, a.part_acc + pv * D, a.part_m + pv,
                       a.part_l + pv);
      } else {
        fp32_vector<D>(p, row, h, g, svs, 0, N, nullptr, nullptr, nullptr);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, L::kTmemCols);
  }
}

}  // namespace pf

// Whether the dense tensor-core prefill serves a shape, and its shared memory.
// It does when head_dim is 128 or 256, the lists are long enough against the
// cache for the dense blocks to pay (4 * max_sel >= N: the masked products
// are at most three times the selected ones), and a tile's row bitmasks fit
// in shared memory.
bool prefill_tc_plan(int D, int G, int rows, long long N, int max_sel, int* smem_bytes,
                     int* mask_rows) {
  if (D != 128 && D != 256) return false;
  if (rows < 1 || N < 1 || max_sel < 1 || N > INT32_MAX / 2) return false;
  if (4LL * max_sel < N) return false;
  const long long mr = std::min<long long>(127 / G + 2, rows);
  const long long nblocks = (N + pf::BN - 1) / pf::BN;
  const long long words = nblocks * (pf::BN / 32);  // ceil(N / 32) rounded up to whole blocks
  const long long mask = ((mr * words * 4 + nblocks + mr) + 15) / 16 * 16;
  const long long base = D == 256 ? pf::Layout<256>::kMask : pf::Layout<128>::kMask;
  const long long total = base + mask;
  if (total > 227 * 1024) return false;
  *smem_bytes = (int)total;
  *mask_rows = (int)mr;
  return true;
}

template <int D, bool STAGED>
static cudaError_t run_prefill_tc(const pf::Args& a, int smem, int tiles, cudaStream_t s) {
  auto kern = pf::prefill_tc_kernel<D, STAGED>;
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(done.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (STAGED) {
    // the operand images and the rows' bitmasks first (their kernel waits
    // for the previous one of the stream; the prefill kernel waits for it)
    cfg.gridDim = dim3((unsigned)(a.p.Hkv * a.nblocks + a.p.rows));
    cfg.blockDim = dim3(pf::kCvtThreads);
    cfg.dynamicSmemBytes = (size_t)(a.mask_words + 2) * 4;
    e = cudaLaunchKernelEx(&cfg, pf::prefill_stage_kernel<D>, a,
                           const_cast<uint8_t*>(a.stage));
    if (e != cudaSuccess) return e;
  }
  cfg.gridDim = dim3((unsigned)(tiles * a.nsplit));
  cfg.blockDim = dim3(pf::Roles<STAGED>::kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess || a.nsplit == 1) return e;
  // the splits' partials merged as the decode's are (the sink, O, lse)
  return launch_combine(a.part_acc, a.part_m, a.part_l, a.p.rows * a.p.Hkv, a.nsplit, a.p.Hq,
                        a.p.Hkv, D, a.p.sink, a.p.out, a.p.lse, s);
}

// The staged form's workspace before the partials: the operand images
// (Hkv x blocks x K and V x 128 x D fp16), every row's bitmask (4 words per
// block) and every row's repeat flag.
static size_t stage_image_bytes(long long N, int Hkv, int D) {
  return (size_t)Hkv * (size_t)((N + pf::BN - 1) / pf::BN) * 2 * pf::BN * D * 2;
}

size_t prefill_stage_bytes(long long N, int Hkv, int D, int rows) {
  if (N < 1 || Hkv < 1 || rows < 1 || (D != 128 && D != 256)) return 0;
  const size_t words = (size_t)((N + pf::BN - 1) / pf::BN) * (pf::BN / 32);
  return stage_image_bytes(N, Hkv, D) + (size_t)rows * words * 4 + (size_t)rows * 4;
}

size_t prefill_partial_bytes(int rows, int Hq, int D, int nsplit) {
  if (nsplit <= 1) return 0;
  return (size_t)rows * Hq * nsplit * ((size_t)D + 2) * 4;
}

int prefill_auto_splits(int rows, int G, int Hkv, int sms) {
  // A tile's blocks split over several CTAs only where the tiles alone would
  // leave more than half of the SMs idle: as many splits as fit one wave (up
  // to 8); otherwise the partials' round trip would cost more than it saves.
  const long long tiles = (((long long)rows * G + pf::BM - 1) / pf::BM) * Hkv;
  if (tiles < 1 || sms < 1 || 2 * tiles > sms) return 1;
  return (int)std::min<long long>(8, sms / tiles);
}

cudaError_t launch_dsa_prefill_tc(const DecodeParams& p, int D, int smem, int mask_rows,
                                  void* stage, int nsplit, float* part, cudaStream_t s) {
  pf::Args a;
  a.p = p;
  a.stage = static_cast<const uint8_t*>(stage);
  a.nsplit = nsplit;
  const long long pvec = (long long)p.rows * p.Hq * nsplit;  // partial vectors
  a.part_acc = nsplit > 1 ? part : nullptr;
  a.part_m = nsplit > 1 ? part + pvec * D : nullptr;
  a.part_l = nsplit > 1 ? part + pvec * (D + 1) : nullptr;
  const long long nvec = (long long)p.rows * p.G;
  a.tiles_per_head = (int)((nvec + pf::BM - 1) / pf::BM);
  a.mask_rows = mask_rows;
  a.nblocks = (int)((p.cache_rows + pf::BN - 1) / pf::BN);
  a.mask_words = a.nblocks * (pf::BN / 32);
  a.gmask = nullptr;
  a.gdup = nullptr;
  if (stage != nullptr) {
    a.gmask = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(stage) +
                                          stage_image_bytes(p.cache_rows, p.Hkv, D));
    a.gdup = reinterpret_cast<int*>(a.gmask + (long long)p.rows * a.mask_words);
  }
  const long long tiles = (long long)a.tiles_per_head * p.Hkv;
  if (tiles * nsplit > INT32_MAX || (long long)a.nblocks * p.Hkv + p.rows > INT32_MAX)
    return cudaErrorInvalidValue;
  if (stage != nullptr)
    return D == 256 ? run_prefill_tc<256, true>(a, smem, (int)tiles, s)
                    : run_prefill_tc<128, true>(a, smem, (int)tiles, s);
  return D == 256 ? run_prefill_tc<256, false>(a, smem, (int)tiles, s)
                  : run_prefill_tc<128, false>(a, smem, (int)tiles, s);
}

}  // namespace i8kv
