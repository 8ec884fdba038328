// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace i8kv {

enum class Path : int { kDsa = 1, kPaged = 2 };

struct DecodeParams {
  const void* q;             // fp16 [rows, Hq, D]
  const void* k;             // cache base (int8 or fp16)
  const void* v;
  const float* k_scale;      // [1] or [Hkv, D]; unused for an fp16 cache
  const float* v_scale;
  const int32_t* idx;        // DSA: [rows, max_sel]
  const int32_t* block_table;  // paged: [rows, max_blocks]
  const int32_t* seq_lens;     // paged: [rows]
  const float* sink;         // [Hq] or nullptr
  void* out;                 // fp16 [rows, Hq, D]
  float* lse;                // [rows, Hq] or nullptr
  float* ws_acc;             // [units, splits, G, D]
  float* ws_m;               // [units, splits, G]
  float* ws_l;               // [units, splits, G]
  int32_t* slots_out;        // paged debug [rows, cap] or nullptr
  uint32_t* flags;           // or nullptr
  int64_t cache_rows;        // DSA: N; paged: num_blocks (in blocks)
  int32_t rows, Hq, Hkv, G;
  int32_t max_sel;           // DSA list length (cap)
  int32_t bs, max_blocks;    // paged
  int32_t bs_log2;           // log2(bs) when bs is a power of two, else -1
  int32_t num_splits, chunk;
  int32_t per_channel;       // 1: scales [Hkv, D]; 0: one scale
  float sigma;
  float softcap;             // paged: > 0 caps scores to softcap * tanh(s / softcap); 0 off
  int32_t window;            // paged: >= 0 attends [len - 1 - window, len); -1 off
  int32_t lpt;               // paged: longest-first dispatch of the (unit, split) items
  // paged, balanced pieces (chunk 0 on the API): the live lengths are cut on
  // the device into pieces of about equal length across the batch, at most
  // num_splits per row (the partial slots), bal_pieces (row, piece) pairs in
  // all, each a multiple of bal_round positions; the grid has
  // ceil(num_splits / 2) CTAs per unit (decode_kernel.cuh, balanced_item)
  int32_t balanced;
  int32_t bal_round;
  int32_t bal_pieces;
};

// Longest-first dispatch of the paged decode (decode_kernel.cuh, lpt_item):
// batches of at most kLptMaxRows rows, chunks of at least kLptMinChunk tokens.
constexpr int kLptMaxRows = 128;
constexpr int kLptMinChunk = 1280;

struct KernelKey {
  Path path;
  int D;
  int nt;          // 8-head tiles: 1 (G <= 8) or 2 (G <= 16)
  bool fp16_cache;
  bool fp8_cache;  // float8 e4m3fn codes (same tile as int8, other conversion)
  bool p_lo;       // probability tile as fp16 high + low parts
};

// What the geometry needs to know of a decode kernel instantiation.
struct KernelInfo {
  int occupancy;  // resident CTAs per SM (the CUDA occupancy API)
  int round;      // positions one round of the CTA's warps covers (warps x step)
};

// Per-path launchers (one per translation unit): grid (rows * Hkv, num_splits);
// with info != NULL nothing is launched and the selected kernel's KernelInfo
// is returned there instead.
cudaError_t launch_dsa_decode(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                              KernelInfo* info);
cudaError_t launch_dsa_prefill(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                               KernelInfo* info);
cudaError_t launch_paged_int8(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                              KernelInfo* info);
cudaError_t launch_paged_fp16(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                              KernelInfo* info);
cudaError_t launch_paged_fp8(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                             KernelInfo* info);

// The dense tensor-core prefill (prefill_tc.cu): whether it serves a shape
// (and with how much shared memory / how many mask rows), and its launch.
bool prefill_tc_plan(int D, int G, int rows, long long N, int max_sel, int* smem_bytes,
                     int* mask_rows);
// stage: NULL for the converting form; else the staged form's operand images
// and row bitmasks (prefill_stage_bytes of them, 16-byte aligned), written by
// the call itself.
// nsplit > 1 (staged form only): each tile's blocks split over nsplit CTAs,
// whose partials (prefill_partial_bytes at part: acc, then m, then l) the
// combine kernel merges into out and lse.
cudaError_t launch_dsa_prefill_tc(const DecodeParams& p, int D, int smem, int mask_rows,
                                  void* stage, int nsplit, float* part, cudaStream_t s);
size_t prefill_stage_bytes(long long N, int Hkv, int D, int rows);
size_t prefill_partial_bytes(int rows, int Hq, int D, int nsplit);
// The automatic split count of the dense prefill on a device with sms SMs.
int prefill_auto_splits(int rows, int G, int Hkv, int sms);

cudaError_t launch_combine(const float* acc, const float* m, const float* l, int units,
                           int num_splits, int Hq, int Hkv, int D, const float* sink, void* out,
                           float* lse, cudaStream_t stream);
cudaError_t launch_int8_to_fp16(const int8_t* in, uint16_t* out, int64_t n, cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const void* k_new, const void* v_new, const int32_t* slots,
                                     int num_tokens, int Hkv, int D, void* k_cache,
                                     void* v_cache, long long num_slots, const float* ks,
                                     const float* vs, int per_channel, bool fp8, uint32_t* flags,
                                     cudaStream_t stream);
cudaError_t launch_fp8_to_fp16(const uint8_t* in, uint16_t* out, int64_t n, cudaStream_t stream);

}  // namespace i8kv
