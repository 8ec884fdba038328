/*
 * int8kv.h -- C ABI of libint8kv.so: split-KV GQA decode attention over an
 * INT8-quantized KV cache on GB300 (sm_103a).
 *
 * The operation (all entry points below compute parts of it):
 *   For each query row r and query head h, with KV head g = h / G and
 *   G = Hq / Hkv (contiguous GQA groups):
 *     K_t = k_scale * code_K[t, g, :]   V_t = v_scale * code_V[t, g, :]
 *         (per-tensor scale: one number; per-channel: scale[g, d])
 *     s_t = softmax_scale * dot(Q[r, h, :], K_t)       (natural-log units)
 *     O[r, h, :] = sum_t exp(s_t - m) V_t / sum_t exp(s_t - m),  m = max_t s_t
 *     lse[r, h]  = m + ln sum_t exp(s_t - m)
 *     optional head sink s_h:  O <- O / (1 + exp(s_h - lse))
 *   over the candidate set of the row: the valid entries of a sparse index
 *   list (onnxruntime PR 33707 "INT8-KV DynamicSparseAttention", Summary of
 *   Changes §1-§2) or the first min(seq_len, cap) tokens of a paged
 *   block-table cache (onnxruntime PR 29912 "PagedAttention: quantized KV
 *   cache ...", CUDA kernels: paged decode, ApplyHeadSink).  The decode calls
 *   split each row's candidates into chunks, run an online softmax per chunk
 *   and merge the partials with a log-sum-exp combine (PR 33707 §2); the split
 *   count comes from the capacity and the row count only (onnx-genai PR 1350
 *   "adaptive split-KV sizing", Summary).
 *
 * Conventions shared by every entry point
 *   - Device pointers are CUDA device addresses of the current device.  The
 *     caller owns every buffer; the library allocates nothing, never
 *     synchronises the host and enqueues work only on `stream` (a
 *     cudaStream_t passed as void*; NULL = the legacy default stream).
 *   - fp16 tensors are passed as uint16_t* (IEEE binary16 bit patterns).
 *   - Layouts are dense row-major with the shapes given per argument.
 *   - Alignment: q, out, caches and per-channel scales must be 16-byte
 *     aligned; index lists, block tables, lengths, lse, sinks and flags
 *     4-byte aligned; the workspace 16-byte aligned.
 *   - Argument errors are reported by the return value before anything is
 *     enqueued.  A launch failure returns I8KV_ECUDA.  Data-dependent
 *     conditions found on the device are OR-ed into the optional `flags`
 *     word (I8KV_FLAG_*) and never stop the kernel.
 *   - Every call with the same shapes and geometry enqueues the same
 *     kernels with the same launch configuration, so calls can be captured
 *     in a CUDA graph; live lengths are read on the device.
 */
#ifndef INT8KV_H_
#define INT8KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
typedef enum {
  I8KV_OK = 0,
  I8KV_EINVAL = 1,        /* bad argument: NULL required pointer, negative size, bad enum,
                             non-finite or negative softmax scale, geometry that misses the cap */
  I8KV_EUNSUPPORTED = 2,  /* valid but not served: head_dim not 64/128/256, G > 16,
                             softmax_scale > 1, block_size not a multiple of 16, ... */
  I8KV_EALIGN = 3,        /* a pointer breaks the alignment rule above */
  I8KV_EWORKSPACE = 4,    /* workspace NULL or smaller than split_workspace_bytes() */
  I8KV_ECUDA = 5          /* a CUDA runtime call or kernel launch failed */
} i8kv_status;

/* ---- enumerations ------------------------------------------------------- */
#define I8KV_SCALE_PER_TENSOR 1  /* k_scale / v_scale: one float                 */
#define I8KV_SCALE_PER_CHANNEL 2 /* k_scale / v_scale: float [Hkv, D]             */

#define I8KV_CACHE_INT8 1 /* codes in [-128, 127], dequantised with the scales */
#define I8KV_CACHE_FP16 2 /* paged_decode only: values taken as is, scales ignored */
#define I8KV_CACHE_FP8 3  /* paged_decode / reshape_and_cache only: float8 e4m3fn codes,
                             dequantised with the scales (onnxruntime PR 29912, Schema:
                             cache element type float8e4m3fn) */

#define I8KV_GEOM_WAVE 0       /* onnx-genai PR 1350 rule (num_splits from one wave)        */
#define I8KV_GEOM_POW2_TILES 1 /* onnxruntime PR 33707 rule (power-of-two tiles per split)  */
#define I8KV_GEOM_BALANCED 2   /* decode_plan, paged path: balanced pieces (see paged_decode) */

#define I8KV_PATH_DSA 1   /* sparse-candidate decode kernel */
#define I8KV_PATH_PAGED 2 /* paged decode kernel            */

#define I8KV_MAX_SPLITS 32 /* at most 32 splits (onnxruntime PR 33707, §2) */

/* bits OR-ed into the optional device `flags` word */
#define I8KV_FLAG_LEN_CLAMPED 0x1u /* a seq_len was > cap (clamped) or < 0 (taken as 0)       */
#define I8KV_FLAG_QUERY_RANGE 0x2u /* some Q*k_scale is not finite or beyond +-65504 (that CTA
                                      took the FP32 path)                                     */
#define I8KV_FLAG_BAD_BLOCK 0x4u   /* a block-table entry inside the live length is outside
                                      [0, num_blocks): those tokens were skipped              */
#define I8KV_FLAG_BAD_SLOT 0x8u    /* reshape_and_cache: a slot >= num_slots was skipped      */
#define I8KV_FLAG_FP32_PATH 0x10u  /* some CTA evaluated its heads on the FP32 path (see the
                                      numerical eligibility rules below)                     */
#define I8KV_FLAG_WAIT_TIMEOUT 0x20u /* dsa_prefill's tensor-core kernel: a CTA gave up waiting
                                        (about a second) for its own asynchronous copies or
                                        tensor-core products; its outputs are NaN          */

/* Human-readable name of a status code (static storage). */
const char* i8kv_status_string(int status);

/* Library ABI version (major*100 + minor).  3.0: dsa_prefill_ws and
 * dsa_prefill_workspace_bytes take num_splits; dsa_prefill_auto_splits. */
int32_t i8kv_version(void);

/* The cudaError_t value behind the calling thread's most recent I8KV_ECUDA
 * (0 if there was none). */
int32_t i8kv_last_cuda_error(void);

/*
 * split_geometry -- pure host integer arithmetic, no CUDA call.
 *
 * Chooses the number of splits and the chunk length (in candidates or tokens)
 * from the capacity `cap` (list length or max_blocks*block_size) and the number
 * of independent work units `units` (rows x KV heads), never from a live length.
 *   mode I8KV_GEOM_WAVE (onnx-genai PR 1350, Summary):
 *     n = min(ceil(wave_ctas / units), ceil(cap / min_chunk), max_splits);
 *     chunk = ceil(cap / n) rounded up to a multiple of `granule`;
 *     n = ceil(cap / chunk).  override_value > 0 pins the chunk instead:
 *     n = min(ceil(cap / override_value), max_splits), then as above.
 *   mode I8KV_GEOM_POW2_TILES (onnxruntime PR 33707, §2): tiles = ceil(cap /
 *     granule); tiles_per_split = smallest power of two with
 *     ceil(tiles / tps) * units <= wave_ctas (override_value > 0: that tps as a
 *     target); n = min(ceil(tiles / tps), max_splits); tiles_eff = ceil(tiles /
 *     n); n = ceil(tiles / tiles_eff); chunk = tiles_eff * granule.
 *   cap <= 0 gives n = 1, chunk = granule.
 * Outputs: *num_splits in [1, max_splits], *chunk a multiple of granule with
 * num_splits * chunk >= cap and (num_splits - 1) * chunk < cap.
 * Errors: I8KV_EINVAL for units, wave_ctas, granule, min_chunk or max_splits < 1,
 * override_value < 0, an unknown mode or NULL outputs.
 */
i8kv_status split_geometry(int64_t cap, int32_t units, int32_t wave_ctas, int32_t granule,
                           int32_t min_chunk, int32_t max_splits, int32_t mode,
                           int32_t override_value, int32_t* num_splits, int32_t* chunk);

/*
 * split_workspace_bytes -- bytes of the split workspace for `units` work units
 * of G query heads of dimension D and `num_splits` splits.  Layout (fp32):
 *   acc [units, num_splits, G, D]   un-normalised partial outputs, value-scaled
 *   m   [units, num_splits, G]      running maximum (natural log)
 *   l   [units, num_splits, G]      running sum of exp(s - m)
 * The partial vectors come first so that they stay 16-byte aligned
 * (onnxruntime PR 33707, §2).  Returns 0 for num_splits <= 1 or bad sizes.
 */
size_t split_workspace_bytes(int32_t units, int32_t num_splits, int32_t G, int32_t D);

/*
 * decode_plan -- the geometry a decode call uses when it is given
 * num_splits = 0 (automatic), for the current device.
 *   path: I8KV_PATH_DSA or I8KV_PATH_PAGED; cache_dtype: I8KV_CACHE_INT8 or
 *   I8KV_CACHE_FP16 (paged only); cap: max_sel (DSA) or max_blocks*block_size
 *   (paged); rows: S (DSA) or B (paged); mode / override_value as in
 *   split_geometry.  wave_ctas = SM count x resident CTAs per SM of the
 *   selected decode kernel (queried from the CUDA occupancy API and cached per
 *   device); granule = 64 (POW2_TILES) or 16 (WAVE); min_chunk = 128;
 *   mode I8KV_GEOM_BALANCED (paged path only, else I8KV_EUNSUPPORTED):
 *   num_splits = min(32, max(2, 2 x the WAVE rule's automatic count)) partial
 *   slots and chunk = 0, for paged_decode's balanced pieces;
 *   max_splits = I8KV_MAX_SPLITS.  For the paged path in WAVE mode with
 *   override_value 0 the chunk is then moved to the multiple of one round of
 *   the paged kernel's CTA (4 warps x its step: 128 positions for an int8 or
 *   e4m3fn cache with head_dim <= 128, else 64) nearer to
 *   ceil(cap / num_splits) -- the lower one only if it is >= 128 and gives at
 *   most I8KV_MAX_SPLITS splits -- and num_splits = ceil(cap / chunk).
 * Outputs: *num_splits, *chunk, *workspace_bytes (0 when one split), and, if
 * wave_ctas is not NULL, the wave used.  Errors as for the decode calls'
 * shape checks, I8KV_ECUDA if the device cannot be queried.
 */
i8kv_status decode_plan(int32_t path, int32_t cache_dtype, int64_t cap, int32_t rows,
                        int32_t Hq, int32_t Hkv, int32_t D, int32_t mode,
                        int32_t override_value, int32_t* num_splits, int32_t* chunk,
                        size_t* workspace_bytes, int32_t* wave_ctas);

/*
 * dsa_decode -- sparse-candidate decode (onnxruntime PR 33707, Summary of
 * Changes §2: split-K decode over a per-row candidate list of an INT8 cache).
 *   q        [S, Hq, D] fp16                 query rows
 *   k_cache  [N, Hkv, D] int8, v_cache same  the main cache (token-major)
 *   k_scale, v_scale, scale_kind             fp32 [1] or [Hkv, D]
 *   idx      [S, max_sel] int32              row r attends the entries of
 *            idx[r, :] that lie in [0, N), in list order, duplicates counted;
 *            any other value is skipped (padding: -1)
 *   softmax_scale                            sigma, 0 <= sigma <= 1 (the FP16
 *            query / probability path is bounded for sigma <= 1: PR 33707 §1)
 *   head_sink [Hq] fp32 or NULL              per-head sink logit (PR 29912)
 *   num_splits, chunk                        geometry: split k of row r covers
 *            list positions [k*chunk, (k+1)*chunk); requires num_splits in
 *            [1, 32], chunk > 0 and a multiple of 16, num_splits*chunk >=
 *            max_sel.  num_splits = 0: automatic (decode_plan, POW2_TILES rule,
 *            chunk ignored).
 *   workspace, workspace_bytes               >= split_workspace_bytes(S*Hkv,
 *            num_splits, G, D) when num_splits > 1 (may be NULL otherwise)
 *   out      [S, Hq, D] fp16                 output.  NULL with num_splits > 1:
 *            write the split partials to the workspace only and enqueue no
 *            combine (the caller runs split_combine later, e.g. after gathering
 *            partials of one row computed on several devices)
 *   lse      [S, Hq] fp32 or NULL            log-sum-exp of the attended scores
 *            (without the sink); -inf for an empty candidate set (O = 0)
 *   flags    device uint32 or NULL           I8KV_FLAG_* bits are OR-ed in
 * Work: one kernel over (S*Hkv units) x num_splits CTAs writing partials, then
 * the split_combine kernel; with one split the decode kernel writes O directly.
 * S = 0 or max_sel = 0 enqueues nothing for S = 0 and writes O = 0, lse = -inf
 * for max_sel = 0.
 */
i8kv_status dsa_decode(const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache,
                       const float* k_scale, const float* v_scale, int32_t scale_kind,
                       const int32_t* idx, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                       int64_t N, int32_t max_sel, float softmax_scale, const float* head_sink,
                       int32_t num_splits, int32_t chunk, void* workspace,
                       size_t workspace_bytes, uint16_t* out, float* lse, uint32_t* flags,
                       void* stream);

/*
 * dsa_prefill -- the tensor-core multi-row variant over gathered candidates
 * (onnxruntime PR 33707, Summary of Changes §1: grid (rows, KV heads), no
 * splits, the probability tile as a single FP16 tile).  Arguments as for
 * dsa_decode without the geometry and the workspace; any S >= 0.
 */
i8kv_status dsa_prefill(const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache,
                        const float* k_scale, const float* v_scale, int32_t scale_kind,
                        const int32_t* idx, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                        int64_t N, int32_t max_sel, float softmax_scale,
                        const float* head_sink, uint16_t* out, float* lse, uint32_t* flags,
                        void* stream);

/*
 * dsa_prefill_workspace_bytes -- bytes of the workspace that lets dsa_prefill_ws
 * take the staged form of the tensor-core kernel for this shape and split
 * count (num_splits as for dsa_prefill_ws; 0 = the automatic count on the
 * current device): Hkv x ceil(N / 128) x 2 x 128 x D x 2 (the cache as fp16
 * operand images) + S x ceil(N / 128) x 16 (every row's candidate bitmask)
 * + S x 4 (every row's repeat flag), plus with more than one split, from the
 * next 256-byte boundary, S x Hq x splits x (D + 2) x 4 (the splits' fp32
 * partials: the accumulators, then m, then l).  0 when the tensor-core kernel does not
 * serve the shape (head_dim other than 128 / 256, 4 * max_sel < N, masks too
 * large for shared memory, S, N or max_sel < 1, bad heads) or num_splits is
 * outside [0, 32].  Host only (the automatic count reads the SM count).
 */
size_t dsa_prefill_workspace_bytes(int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int64_t N,
                                   int32_t max_sel, int32_t num_splits);

/*
 * dsa_prefill_auto_splits -- the automatic split count of the tensor-core
 * prefill (num_splits = 0) on a device with `sms` SMs: with tiles = Hkv x
 * ceil(S x (Hq / Hkv) / 128) tiles of 128 (row, head) vectors, min(8, sms /
 * tiles) where 2 x tiles <= sms, else 1 (a split's partials cost a round trip
 * through the combine kernel, paid back only where tiles leave SMs idle).
 * 0 for S < 1, sms < 1 or bad heads.  Host arithmetic only.
 */
int32_t dsa_prefill_auto_splits(int32_t S, int32_t Hq, int32_t Hkv, int32_t sms);

/*
 * dsa_prefill_ws -- dsa_prefill with an optional workspace (the caller's device
 * memory, 16-byte aligned, workspace_bytes >= dsa_prefill_workspace_bytes for
 * the same num_splits).  With one, where the tensor-core kernel serves the
 * shape, the call first converts the cache once into fp16 operand images in
 * the workspace (a kernel of its own, about 3 bytes written per cache byte
 * read, whose other CTAs also turn each row's list into a bitmask of cache
 * positions) and the prefill kernel copies each block in with one bulk copy
 * instead of converting it in every CTA; unsplit, the results are the same
 * bit for bit.
 *   num_splits  0: automatic -- where a KV head's tiles of 128 (row, head)
 *               vectors number fewer than half the SMs, each tile's blocks
 *               are split over min(8, SMs / tiles) CTAs, else 1;
 *               1 .. 32: that many (a split may get no block).
 *               With more than one, each CTA writes the fp32 partials of its
 *               share of the tile's blocks (and of the candidates at their
 *               positions; a vector sent to the FP32 path publishes an FP32
 *               partial of its share), and the split_combine kernel merges
 *               them with the sink into out and lse (onnxruntime PR 33707,
 *               Summary of Changes §2: the split-K partials and their merge).
 * With workspace NULL, or where the gathering kernel serves the shape, it is
 * dsa_prefill (unsplit; num_splits has no effect on the gathering kernel).
 * The workspace holds nothing the caller needs afterwards.
 * Errors: as dsa_prefill; I8KV_EINVAL if num_splits is outside [0, 32];
 * I8KV_EWORKSPACE if workspace_bytes is too small, or workspace is NULL with
 * num_splits > 1 on the tensor-core path; I8KV_EALIGN if the workspace is not
 * 16-byte aligned.
 */
i8kv_status dsa_prefill_ws(const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache,
                           const float* k_scale, const float* v_scale, int32_t scale_kind,
                           const int32_t* idx, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                           int64_t N, int32_t max_sel, float softmax_scale,
                           const float* head_sink, int32_t num_splits, void* workspace,
                           size_t workspace_bytes, uint16_t* out, float* lse, uint32_t* flags,
                           void* stream);

/*
 * paged_decode -- split-KV decode over a paged block-table cache
 * (onnxruntime PR 29912, CUDA kernels: "split-KV, block-table-aware decode
 * with native head-sink ... and on-the-fly cache dequantization").
 *   q            [B, Hq, D] fp16              one query row per sequence
 *   k_cache, v_cache [num_blocks, block_size, Hkv, D] int8, float8 e4m3fn or fp16
 *   cache_dtype  I8KV_CACHE_INT8, I8KV_CACHE_FP8 (both dequantised with the
 *                scales) or I8KV_CACHE_FP16 (scales ignored, may be NULL)
 *   block_table  [B, max_blocks] int32        token t of sequence b is row
 *                block_table[b, t / block_size] * block_size + t % block_size
 *   seq_lens     [B] int32, DEVICE memory     live lengths, clamped to
 *                cap = max_blocks * block_size (I8KV_FLAG_LEN_CLAMPED)
 *   block_size   a multiple of 16
 *   num_splits, chunk  as for dsa_decode over token positions, with cap =
 *                max_blocks*block_size; num_splits = 0: automatic (WAVE rule).
 *                num_splits in [2, 32] with chunk = 0: balanced pieces (not on
 *                the pages; decode_plan's I8KV_GEOM_BALANCED gives the values):
 *                num_splits partial slots per row and ceil(num_splits / 2)
 *                CTAs per (row, KV head), all fixed by the arguments, while
 *                each CTA cuts its piece of a row's live range on the device
 *                from all live lengths, so that the pieces are about equally
 *                long across a ragged batch (about one occupancy wave of
 *                them); the combine merges the used slots, the others are
 *                marked empty.  Needs B <= 128 and slots_out NULL
 *                (I8KV_EUNSUPPORTED otherwise).
 *   slots_out    [B, cap] int32 or NULL       debug output: the gathered row of
 *                every token position, -1 past the live length
 *   other arguments as for dsa_decode.
 */
i8kv_status paged_decode(const uint16_t* q, const void* k_cache, const void* v_cache,
                         int32_t cache_dtype, const float* k_scale, const float* v_scale,
                         int32_t scale_kind, const int32_t* block_table,
                         const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t block_size, int32_t max_blocks, int64_t num_blocks,
                         float softmax_scale, const float* head_sink, int32_t num_splits,
                         int32_t chunk, void* workspace, size_t workspace_bytes, uint16_t* out,
                         float* lse, int32_t* slots_out, uint32_t* flags, void* stream);

/*
 * paged_decode_ex -- paged_decode with the two score options the same page
 * lists for that kernel (onnxruntime PR 29912, CUDA kernels: "native head-sink,
 * softcap, sliding-window and on-the-fly cache dequantization").  The page
 * names them without a definition; the meanings taken are:
 *   softcap  >= 0, finite.  > 0: each scaled score s becomes
 *            softcap * tanh(s / softcap) before the softmax; 0: off.  The
 *            head-sink logit is not capped.
 *   window   >= -1.  >= 0: the query of sequence b (at position L - 1, L its
 *            clamped live length) attends positions [max(0, L-1-window), L):
 *            itself and the window positions before it; -1: off.
 * With a window the splits count their chunks from the window start rounded
 * down to a multiple of 16, and num_splits * chunk must cover
 * I8KV_WINDOW_SPAN(cap, window) (not cap); num_splits = 0 plans over that span
 * (decode_plan with cap = I8KV_WINDOW_SPAN(cap, window) gives the same
 * geometry).  slots_out then holds -1 outside the window.  Other arguments,
 * errors and work as for paged_decode; softcap < 0, non-finite, or
 * window < -1 -> I8KV_EINVAL.
 */
#define I8KV_WINDOW_SPAN(cap, window)                                              \
  ((window) < 0 || (int64_t)(cap) <= (int64_t)(window) + 16 ? (int64_t)(cap)      \
                                                            : (int64_t)(window) + 16)

/* paged_window_span -- I8KV_WINDOW_SPAN(cap, window) as a function, for
 * bindings that cannot expand the macro: the positions a windowed paged decode's
 * splits cover (cap when window < 0).  Pure host arithmetic, no CUDA call. */
int64_t paged_window_span(int64_t cap, int32_t window);

i8kv_status paged_decode_ex(const uint16_t* q, const void* k_cache, const void* v_cache,
                            int32_t cache_dtype, const float* k_scale, const float* v_scale,
                            int32_t scale_kind, const int32_t* block_table,
                            const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv,
                            int32_t D, int32_t block_size, int32_t max_blocks, int64_t num_blocks,
                            float softmax_scale, const float* head_sink, float softcap,
                            int32_t window, int32_t num_splits, int32_t chunk, void* workspace,
                            size_t workspace_bytes, uint16_t* out, float* lse,
                            int32_t* slots_out, uint32_t* flags, void* stream);

/*
 * split_combine -- log-sum-exp merge of split partials plus the head sink
 * (onnxruntime PR 33707 §2: the merge kernel; PR 29912: ApplyHeadSink):
 *   M = max_k m_k;  L = sum_k l_k exp(m_k - M);  O = sum_k acc_k exp(m_k - M) / L
 *   lse = M + ln L;  O <- O / (1 + exp(s_h - lse)) if a sink is given.
 * Splits with m_k = -inf are skipped (their acc is not read); all skipped:
 * O = 0, lse = -inf.
 *   acc [units, num_splits, G, D], m, l [units, num_splits, G] fp32 (the
 *   workspace layout of split_workspace_bytes); unit u = row * Hkv + g;
 *   G = Hq / Hkv; out [units*G, D] fp16 (= [rows, Hq, D]); lse [units*G] or
 *   NULL; head_sink [Hq] or NULL, indexed by h = (u % Hkv) * G + j.
 *   num_splits in [1, 32]; D in {64, 128, 256}.
 */
i8kv_status split_combine(const float* acc, const float* m, const float* l, int32_t units,
                          int32_t num_splits, int32_t Hq, int32_t Hkv, int32_t D,
                          const float* head_sink, uint16_t* out, float* lse, void* stream);

/*
 * reshape_and_cache -- quantize-on-write of new key / value rows into a paged
 * INT8 or float8 e4m3fn cache (onnxruntime PR 29912, CUDA kernels:
 * "ReshapeAndCache quantizes on write"; Schema: cache element type int8 or
 * float8e4m3fn).  For every new token n and KV head g, the cache row
 * (slot_mapping[n], g) receives, with q = x[d] / scale:
 *     I8KV_CACHE_INT8: code[d] = clamp(round_half_even(q), -127, 127)
 *     I8KV_CACHE_FP8:  code[d] = the e4m3fn value nearest q (ties to even),
 *                      saturated to +-448
 * with scale = k_scale / v_scale per tensor ([1]) or per channel ([Hkv, D]); q
 * is the IEEE fp32 quotient of the fp16 value widened to fp32 (exactly: the
 * kernel's faster product by the reciprocal falls back to the division
 * wherever the two could round differently); a NaN quotient stores 0.
 *   k_new, v_new   [num_tokens, Hkv, D] fp16, device
 *   slot_mapping   [num_tokens] int32, device: row of the flattened cache
 *                  (block * block_size + offset); < 0: skipped (padding);
 *                  >= num_slots: skipped and I8KV_FLAG_BAD_SLOT raised
 *   k_cache, v_cache [num_slots, Hkv, D] bytes (a paged cache [num_blocks,
 *                  block_size, Hkv, D] with num_slots = num_blocks * block_size)
 *   cache_dtype    I8KV_CACHE_INT8 or I8KV_CACHE_FP8 (others: I8KV_EINVAL)
 *   D a multiple of 8; caches, rows and per-channel scales 16-byte aligned.
 * Scales must be finite and positive (not checked on the device).
 */
i8kv_status reshape_and_cache(const uint16_t* k_new, const uint16_t* v_new,
                              const int32_t* slot_mapping, int32_t num_tokens, int32_t Hkv,
                              int32_t D, void* k_cache, void* v_cache, int64_t num_slots,
                              const float* k_scale, const float* v_scale, int32_t scale_kind,
                              int32_t cache_dtype, uint32_t* flags, void* stream);

/*
 * dsa_decode_static_workspace -- dsa_decode without a caller-supplied
 * workspace, for callers that cannot allocate device memory when they call
 * (an engine's enqueue step that must not allocate, code with no access to the
 * application's allocator, loops that must never enter the allocator).  The
 * pages have no counterpart; this is a convenience of this library.
 *   Arguments and results as for dsa_decode, without workspace and
 *   workspace_bytes, except that out must not be NULL when S > 0 (I8KV_EINVAL:
 *   partials left in the library's private array could not be read by the
 *   caller).  The split partials go to a device array inside the
 *   library of I8KV_STATIC_WORKSPACE_BYTES bytes, allocated when CUDA loads the
 *   library's device code on a device and held on every such device until the
 *   process exits.  Nothing is allocated or freed by the call itself.
 *   - A geometry whose partials need more than I8KV_STATIC_WORKSPACE_BYTES
 *     (split_workspace_bytes(S*Hkv, num_splits, G, D)) returns
 *     I8KV_EWORKSPACE before anything is enqueued.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current) and caches it; make that
 *     first call before any stream capture.  The cached address belongs to the
 *     device's current CUDA context: do not call this entry point again after
 *     cudaDeviceReset (or any other teardown of the primary context) in the
 *     same process.
 *   - All calls on a device share the one array.  Calls whose kernels can run
 *     at the same time on the GPU (different streams without ordering between
 *     them) race on it and give wrong results; calls ordered on one stream are
 *     fine.  Nothing in it needs clearing between calls: each call's decode
 *     kernel writes the (m, l) entry of every (unit, split, head) that its
 *     combine reads, and the combine reads a split's partial vector only when
 *     that split wrote it.
 */
#define I8KV_STATIC_WORKSPACE_BYTES (4u * 1024u * 1024u)
i8kv_status dsa_decode_static_workspace(const uint16_t* q, const int8_t* k_cache,
                                        const int8_t* v_cache, const float* k_scale,
                                        const float* v_scale, int32_t scale_kind,
                                        const int32_t* idx, int32_t S, int32_t Hq, int32_t Hkv,
                                        int32_t D, int64_t N, int32_t max_sel,
                                        float softmax_scale, const float* head_sink,
                                        int32_t num_splits, int32_t chunk, uint16_t* out,
                                        float* lse, uint32_t* flags, void* stream);

/*
 * int8_to_fp16 -- the decode kernels' in-register int8 -> fp16 conversion
 * applied to a buffer (byte permutes into the mantissa of 1024 + 128, then one
 * fp16x2 subtraction of 1152: exact for all 256 codes; onnxruntime PR 29912,
 * "int8->fp16 conversion fast path").  in [n] int8, out [n] fp16, n a multiple
 * of 4, both 16-byte aligned.  For tests of the conversion.
 */
i8kv_status int8_to_fp16(const int8_t* in, uint16_t* out, int64_t n, void* stream);

/*
 * fp8_to_fp16 -- the paged decode kernel's float8 e4m3fn -> fp16 conversion
 * (cvt.rn.f16x2.e4m3x2, exact) over a device buffer of n codes, n a multiple of
 * 4, both buffers 16-byte aligned; out[i] is the value of in[i] (NaN for the
 * two NaN patterns).  Exposed so that the conversion can be checked
 * exhaustively.
 */
i8kv_status fp8_to_fp16(const uint8_t* in, uint16_t* out, int64_t n, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* INT8KV_H_ */
