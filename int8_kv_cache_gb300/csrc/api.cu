// The extern "C" entry points of libint8kv.so (declared in include/int8kv.h):
// argument validation, split geometry, workspace layout and kernel launches.
// Nothing here allocates device memory or synchronises the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/int8kv.h"
#include "internal.h"

namespace {

using i8kv::DecodeParams;
using i8kv::KernelInfo;
using i8kv::KernelKey;
using i8kv::Path;

thread_local int g_last_cuda_error = 0;

i8kv_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return I8KV_ECUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool supported_head_dim(int32_t D) { return D == 64 || D == 128 || D == 256; }

// Shape checks shared by the decode / prefill calls.
i8kv_status check_heads(int32_t Hq, int32_t Hkv, int32_t D) {
  if (Hq < 1 || Hkv < 1 || D < 1) return I8KV_EINVAL;
  if (Hq % Hkv != 0) return I8KV_EINVAL;
  if (!supported_head_dim(D)) return I8KV_EUNSUPPORTED;
  if (Hq / Hkv > 16) return I8KV_EUNSUPPORTED;
  return I8KV_OK;
}

i8kv_status check_sigma(float s) {
  if (!std::isfinite(s) || s < 0.f) return I8KV_EINVAL;
  if (s > 1.f) return I8KV_EUNSUPPORTED;  // the FP16 path is bounded for scale <= 1 only
  return I8KV_OK;
}

i8kv_status check_scales(const float* ks, const float* vs, int32_t kind) {
  if (kind != I8KV_SCALE_PER_TENSOR && kind != I8KV_SCALE_PER_CHANNEL) return I8KV_EINVAL;
  if (ks == nullptr || vs == nullptr) return I8KV_EINVAL;
  const uintptr_t a = kind == I8KV_SCALE_PER_CHANNEL ? 16 : 4;
  if (!aligned(ks, a) || !aligned(vs, a)) return I8KV_EALIGN;
  return I8KV_OK;
}

KernelKey make_key(Path path, int32_t D, int32_t G, int32_t cache_dtype, bool p_lo) {
  KernelKey k;
  k.path = path;
  k.D = D;
  k.nt = G <= 8 ? 1 : 2;
  k.fp16_cache = cache_dtype == I8KV_CACHE_FP16;
  k.fp8_cache = cache_dtype == I8KV_CACHE_FP8;
  k.p_lo = p_lo;
  return k;
}

cudaError_t launch_key(const KernelKey& key, const DecodeParams& p, cudaStream_t s,
                       KernelInfo* info) {
  if (key.path == Path::kDsa) {
    return key.p_lo ? i8kv::launch_dsa_decode(key, p, s, info)
                    : i8kv::launch_dsa_prefill(key, p, s, info);
  }
  if (key.fp16_cache) return i8kv::launch_paged_fp16(key, p, s, info);
  if (key.fp8_cache) return i8kv::launch_paged_fp8(key, p, s, info);
  return i8kv::launch_paged_int8(key, p, s, info);
}

// One occupancy wave (SM count x resident CTAs per SM) of a kernel on the
// current device and the positions of one round of its CTA, cached per
// (device, kernel).
struct WaveInfo {
  int32_t wave;
  int32_t round;
};

i8kv_status wave_of(const KernelKey& key, WaveInfo* out) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int, int, int>, WaveInfo> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const auto k = std::make_tuple(dev, static_cast<int>(key.path), key.D, key.nt,
                                 static_cast<int>(key.fp16_cache), static_cast<int>(key.fp8_cache),
                                 static_cast<int>(key.p_lo));
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(k);
    if (it != cache.end()) {
      *out = it->second;
      return I8KV_OK;
    }
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DecodeParams dummy{};
  KernelInfo info{0, 0};
  e = launch_key(key, dummy, nullptr, &info);
  if (e != cudaSuccess) return cuda_fail(e);
  const WaveInfo w{std::max(1, sms * std::max(info.occupancy, 1)), std::max(info.round, 16)};
  {
    std::lock_guard<std::mutex> lock(mu);
    cache[k] = w;
  }
  *out = w;
  return I8KV_OK;
}

// SMs of the current device (cached per device).
i8kv_status sm_count(int* sms) {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) {
      *sms = it->second;
      return I8KV_OK;
    }
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> lock(mu);
  cache[dev] = n;
  *sms = n;
  return I8KV_OK;
}

// The dense prefill's split count: num_splits (1 .. I8KV_MAX_SPLITS), or with 0
// the automatic count on the current device.
i8kv_status prefill_splits(int32_t S, int32_t G, int32_t Hkv, int32_t num_splits, int* ns) {
  if (num_splits > 0) {
    *ns = num_splits;
    return I8KV_OK;
  }
  int sms = 0;
  const i8kv_status st = sm_count(&sms);
  if (st != I8KV_OK) return st;
  *ns = i8kv::prefill_auto_splits(S, G, Hkv, sms);
  return I8KV_OK;
}

// The staged prefill's workspace: the operand images and the rows' bitmasks,
// then (with splits) the partials at the next 256-byte boundary.
size_t prefill_ws_bytes(int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int64_t N, int ns) {
  const size_t stage = i8kv::prefill_stage_bytes(N, Hkv, D, S);
  if (ns <= 1) return stage;
  return (stage + 255) / 256 * 256 + i8kv::prefill_partial_bytes(S, Hq, D, ns);
}

constexpr int32_t kGranuleWave = 16;   // the kernels' 16-position MMA tile
constexpr int32_t kGranuleTiles = 64;  // the pages' 64-candidate tile
constexpr int32_t kMinChunk = 128;     // MIN_CHUNK of the wave rule

// The paged decode kernel deals a split's steps (16 or 32 positions) to its 4
// warps in turn, so a chunk that is not a multiple of one round (warps x step:
// 64 or 128 positions) leaves some warps a step, and an HBM round trip, longer
// than the rest.  The automatic wave-rule chunk ceil(cap / n) therefore goes
// to the multiple of the round nearer to it (the lower one only while it stays
// >= MIN_CHUNK and within MAX_SPLITS), and n follows as ceil(cap / chunk).
// Still a function of cap, units and the kernel only.
void snap_to_round(int64_t cap, int64_t round, int32_t* ns, int32_t* chunk) {
  const int64_t raw = cdiv(cap, *ns);
  const int64_t up = cdiv(raw, round) * round;
  const int64_t dn = raw / round * round;
  int64_t ch = up;
  if (dn >= kMinChunk && raw - dn < up - raw && cdiv(cap, dn) <= I8KV_MAX_SPLITS) ch = dn;
  if (ch > INT32_MAX) return;
  *chunk = static_cast<int32_t>(ch);
  *ns = static_cast<int32_t>(cdiv(cap, ch));
}

i8kv_status plan(const KernelKey& key, int64_t cap, int32_t units, int32_t mode, int32_t ovr,
                 int32_t* ns, int32_t* chunk, int32_t* wave_out) {
  WaveInfo w{0, 0};
  i8kv_status st = wave_of(key, &w);
  if (st != I8KV_OK) return st;
  if (wave_out) *wave_out = w.wave;
  const int32_t granule = mode == I8KV_GEOM_POW2_TILES ? kGranuleTiles : kGranuleWave;
  st = split_geometry(cap, units, w.wave, granule, kMinChunk, I8KV_MAX_SPLITS, mode, ovr, ns,
                      chunk);
  if (st != I8KV_OK) return st;
  if (key.path == Path::kPaged && mode == I8KV_GEOM_WAVE && ovr == 0 && cap > 0 && *ns > 1)
    snap_to_round(cap, w.round, ns, chunk);
  return I8KV_OK;
}

// Geometry given by the caller: num_splits in [1, 32], chunk a positive
// multiple of 16 with num_splits * chunk >= cap.
// span: the positions the splits must cover (cap, or the window span);
// base_max: the largest first position of split 0 (0, or cap with a window).
i8kv_status check_geometry(int64_t span, int32_t ns, int32_t chunk, int64_t base_max = 0) {
  if (ns < 1 || ns > I8KV_MAX_SPLITS) return I8KV_EINVAL;
  if (chunk < 16 || chunk % 16 != 0) return I8KV_EINVAL;
  if (static_cast<int64_t>(ns) * chunk < span) return I8KV_EINVAL;
  // positions are 32-bit on the device
  if (base_max + static_cast<int64_t>(ns) * chunk > INT32_MAX) return I8KV_EINVAL;
  return I8KV_OK;
}

i8kv_status set_workspace(DecodeParams& p, void* ws, size_t ws_bytes, int32_t units, int32_t ns,
                          int32_t G, int32_t D) {
  p.ws_acc = p.ws_m = p.ws_l = nullptr;
  if (ns <= 1) return I8KV_OK;
  const size_t need = split_workspace_bytes(units, ns, G, D);
  if (ws == nullptr || ws_bytes < need) return I8KV_EWORKSPACE;
  if (!aligned(ws, 16)) return I8KV_EALIGN;
  float* base = static_cast<float*>(ws);
  const size_t nacc = static_cast<size_t>(units) * ns * G * D;
  const size_t nml = static_cast<size_t>(units) * ns * G;
  p.ws_acc = base;
  p.ws_m = base + nacc;
  p.ws_l = base + nacc + nml;
  return I8KV_OK;
}

i8kv_status run(const KernelKey& key, const DecodeParams& p, cudaStream_t s) {
  cudaError_t e = launch_key(key, p, s, nullptr);
  if (e != cudaSuccess) return cuda_fail(e);
  if (p.num_splits > 1 && p.out != nullptr) {
    e = i8kv::launch_combine(p.ws_acc, p.ws_m, p.ws_l, p.rows * p.Hkv, p.num_splits, p.Hq, p.Hkv,
                             key.D, p.sink, p.out, p.lse, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return I8KV_OK;
}

// Common checks of the sparse-candidate calls; fills the shape part of p.
i8kv_status dsa_common(const uint16_t* q, const int8_t* k, const int8_t* v, const float* ks,
                       const float* vs, int32_t kind, const int32_t* idx, int32_t S, int32_t Hq,
                       int32_t Hkv, int32_t D, int64_t N, int32_t max_sel, float sigma,
                       const float* sink, uint16_t* out, float* lse, uint32_t* flags,
                       DecodeParams& p) {
  if (S < 0 || N < 0 || max_sel < 0) return I8KV_EINVAL;
  i8kv_status st = check_heads(Hq, Hkv, D);
  if (st != I8KV_OK) return st;
  if ((st = check_sigma(sigma)) != I8KV_OK) return st;
  if ((st = check_scales(ks, vs, kind)) != I8KV_OK) return st;
  if (S > 0 && (q == nullptr || k == nullptr || v == nullptr)) return I8KV_EINVAL;
  if (S > 0 && max_sel > 0 && idx == nullptr) return I8KV_EINVAL;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k, 16) || !aligned(v, 16)) return I8KV_EALIGN;
  if (!aligned(idx, 4) || !aligned(lse, 4) || !aligned(sink, 4) || !aligned(flags, 4)) return I8KV_EALIGN;
  p = DecodeParams{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.k_scale = ks;
  p.v_scale = vs;
  p.per_channel = kind == I8KV_SCALE_PER_CHANNEL;
  p.idx = idx;
  p.sink = sink;
  p.out = out;
  p.lse = lse;
  p.flags = flags;
  p.cache_rows = N;
  p.rows = S;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.max_sel = max_sel;
  p.sigma = sigma;
  p.softcap = 0.f;
  p.window = -1;
  p.lpt = 0;
  return I8KV_OK;
}

}  // namespace

extern "C" {

const char* i8kv_status_string(int status) {
  switch (status) {
    case I8KV_OK: return "ok";
    case I8KV_EINVAL: return "invalid argument";
    case I8KV_EUNSUPPORTED: return "unsupported shape or option";
    case I8KV_EALIGN: return "misaligned pointer";
    case I8KV_EWORKSPACE: return "workspace missing or too small";
    case I8KV_ECUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int32_t i8kv_version(void) { return 300; }

// The CUDA error code behind the calling thread's last I8KV_ECUDA (0 if none).
int32_t i8kv_last_cuda_error(void) { return g_last_cuda_error; }

int64_t paged_window_span(int64_t cap, int32_t window) { return I8KV_WINDOW_SPAN(cap, window); }

i8kv_status split_geometry(int64_t cap, int32_t units, int32_t wave_ctas, int32_t granule,
                           int32_t min_chunk, int32_t max_splits, int32_t mode,
                           int32_t override_value, int32_t* num_splits, int32_t* chunk) {
  if (num_splits == nullptr || chunk == nullptr) return I8KV_EINVAL;
  if (units < 1 || wave_ctas < 1 || granule < 1 || min_chunk < 1 || max_splits < 1 ||
      override_value < 0)
    return I8KV_EINVAL;
  if (mode != I8KV_GEOM_WAVE && mode != I8KV_GEOM_POW2_TILES) return I8KV_EINVAL;
  if (cap <= 0) {
    *num_splits = 1;
    *chunk = granule;
    return I8KV_OK;
  }
  int64_t n = 0, ch = 0;
  if (mode == I8KV_GEOM_WAVE) {
    if (override_value > 0) {
      n = std::min<int64_t>(cdiv(cap, override_value), max_splits);
    } else {
      const int64_t target = cdiv(wave_ctas, units);
      n = std::min<int64_t>(std::min<int64_t>(target, cdiv(cap, min_chunk)), max_splits);
    }
    n = std::max<int64_t>(n, 1);
    ch = cdiv(cdiv(cap, n), granule) * granule;
    n = cdiv(cap, ch);
  } else {
    const int64_t tiles = cdiv(cap, granule);
    int64_t tps = 1;
    if (override_value > 0) {
      tps = override_value;
    } else {
      while (cdiv(tiles, tps) * units > wave_ctas && tps < tiles) tps *= 2;
    }
    n = std::max<int64_t>(1, std::min<int64_t>(cdiv(tiles, tps), max_splits));
    const int64_t te = cdiv(tiles, n);
    n = cdiv(tiles, te);
    ch = te * granule;
  }
  if (ch > INT32_MAX) return I8KV_EINVAL;
  *num_splits = static_cast<int32_t>(n);
  *chunk = static_cast<int32_t>(ch);
  return I8KV_OK;
}

size_t split_workspace_bytes(int32_t units, int32_t num_splits, int32_t G, int32_t D) {
  if (num_splits <= 1 || units < 1 || G < 1 || D < 1) return 0;
  return static_cast<size_t>(units) * num_splits * G * (static_cast<size_t>(D) + 2) * sizeof(float);
}

i8kv_status decode_plan(int32_t path, int32_t cache_dtype, int64_t cap, int32_t rows, int32_t Hq,
                        int32_t Hkv, int32_t D, int32_t mode, int32_t override_value,
                        int32_t* num_splits, int32_t* chunk, size_t* workspace_bytes,
                        int32_t* wave_ctas) {
  if (num_splits == nullptr || chunk == nullptr || workspace_bytes == nullptr) return I8KV_EINVAL;
  if (path != I8KV_PATH_DSA && path != I8KV_PATH_PAGED) return I8KV_EINVAL;
  if (cache_dtype != I8KV_CACHE_INT8 && cache_dtype != I8KV_CACHE_FP16 &&
      cache_dtype != I8KV_CACHE_FP8)
    return I8KV_EINVAL;
  if (path == I8KV_PATH_DSA && cache_dtype != I8KV_CACHE_INT8) return I8KV_EUNSUPPORTED;
  if (rows < 0 || cap < 0) return I8KV_EINVAL;
  i8kv_status st = check_heads(Hq, Hkv, D);
  if (st != I8KV_OK) return st;
  const int32_t G = Hq / Hkv;
  const KernelKey key = make_key(path == I8KV_PATH_DSA ? Path::kDsa : Path::kPaged, D, G,
                                 cache_dtype, true);
  const int32_t units = std::max(1, rows * Hkv);
  if (mode == I8KV_GEOM_BALANCED) {
    // balanced pieces: twice the wave rule's splits as partial slots (at most
    // MAX_SPLITS), chunk 0 (the pieces are cut on the device)
    if (path != I8KV_PATH_PAGED) return I8KV_EUNSUPPORTED;
    if ((st = plan(key, cap, units, I8KV_GEOM_WAVE, 0, num_splits, chunk, wave_ctas)) != I8KV_OK)
      return st;
    *num_splits = std::min<int32_t>(I8KV_MAX_SPLITS, std::max<int32_t>(2, 2 * *num_splits));
    *chunk = 0;
  } else if ((st = plan(key, cap, units, mode, override_value, num_splits, chunk, wave_ctas)) !=
             I8KV_OK) {
    return st;
  }
  *workspace_bytes = split_workspace_bytes(rows * Hkv, *num_splits, G, D);
  return I8KV_OK;
}

i8kv_status dsa_decode(const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache,
                       const float* k_scale, const float* v_scale, int32_t scale_kind,
                       const int32_t* idx, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                       int64_t N, int32_t max_sel, float softmax_scale, const float* head_sink,
                       int32_t num_splits, int32_t chunk, void* workspace,
                       size_t workspace_bytes, uint16_t* out, float* lse, uint32_t* flags,
                       void* stream) {
  DecodeParams p;
  i8kv_status st = dsa_common(q, k_cache, v_cache, k_scale, v_scale, scale_kind, idx, S, Hq, Hkv,
                              D, N, max_sel, softmax_scale, head_sink, out, lse, flags, p);
  if (st != I8KV_OK) return st;
  if (num_splits < 0) return I8KV_EINVAL;
  const KernelKey key = make_key(Path::kDsa, D, p.G, I8KV_CACHE_INT8, true);
  if (num_splits == 0) {
    st = plan(key, max_sel, std::max(1, S * Hkv), I8KV_GEOM_POW2_TILES, 0, &num_splits, &chunk,
              nullptr);
    if (st != I8KV_OK) return st;
  } else if ((st = check_geometry(max_sel, num_splits, chunk)) != I8KV_OK) {
    return st;
  }
  if ((st = set_workspace(p, workspace, workspace_bytes, S * Hkv, num_splits, p.G, D)) != I8KV_OK)
    return st;
  if (out == nullptr && num_splits == 1 && S > 0) return I8KV_EINVAL;  // nowhere to write
  if (S == 0) return I8KV_OK;
  p.num_splits = num_splits;
  p.chunk = chunk;
  return run(key, p, static_cast<cudaStream_t>(stream));
}

i8kv_status dsa_prefill(const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache,
                        const float* k_scale, const float* v_scale, int32_t scale_kind,
                        const int32_t* idx, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                        int64_t N, int32_t max_sel, float softmax_scale,
                        const float* head_sink, uint16_t* out, float* lse, uint32_t* flags,
                        void* stream) {
  return dsa_prefill_ws(q, k_cache, v_cache, k_scale, v_scale, scale_kind, idx, S, Hq, Hkv, D, N,
                        max_sel, softmax_scale, head_sink, 0, nullptr, 0, out, lse, flags, stream);
}

int32_t dsa_prefill_auto_splits(int32_t S, int32_t Hq, int32_t Hkv, int32_t sms) {
  if (S < 1 || sms < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return 0;
  return i8kv::prefill_auto_splits(S, Hq / Hkv, Hkv, sms);
}

size_t dsa_prefill_workspace_bytes(int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int64_t N,
                                   int32_t max_sel, int32_t num_splits) {
  if (S < 1 || N < 1 || max_sel < 1 || check_heads(Hq, Hkv, D) != I8KV_OK) return 0;
  if (num_splits < 0 || num_splits > I8KV_MAX_SPLITS) return 0;
  int smem = 0, mask_rows = 0;
  if (!i8kv::prefill_tc_plan(D, Hq / Hkv, S, N, max_sel, &smem, &mask_rows)) return 0;
  int ns = 1;
  if (prefill_splits(S, Hq / Hkv, Hkv, num_splits, &ns) != I8KV_OK) return 0;
  return prefill_ws_bytes(S, Hq, Hkv, D, N, ns);
}

i8kv_status dsa_prefill_ws(const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache,
                           const float* k_scale, const float* v_scale, int32_t scale_kind,
                           const int32_t* idx, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                           int64_t N, int32_t max_sel, float softmax_scale,
                           const float* head_sink, int32_t num_splits, void* workspace,
                           size_t workspace_bytes, uint16_t* out, float* lse, uint32_t* flags,
                           void* stream) {
  DecodeParams p;
  i8kv_status st = dsa_common(q, k_cache, v_cache, k_scale, v_scale, scale_kind, idx, S, Hq, Hkv,
                              D, N, max_sel, softmax_scale, head_sink, out, lse, flags, p);
  if (st != I8KV_OK) return st;
  if (S > 0 && out == nullptr) return I8KV_EINVAL;
  if (num_splits < 0 || num_splits > I8KV_MAX_SPLITS) return I8KV_EINVAL;
  if (!aligned(workspace, 16)) return I8KV_EALIGN;
  if (S == 0) return I8KV_OK;
  p.num_splits = 1;
  p.chunk = static_cast<int32_t>(std::max<int64_t>(16, cdiv(max_sel, 16) * 16));
  // dense tensor-core kernel where the rows' lists cover the cache densely
  // enough (a shape rule, so eager and captured calls choose alike), else the
  // gathering mma.sync kernel
  int smem = 0, mask_rows = 0;
  if (i8kv::prefill_tc_plan(D, p.G, S, N, max_sel, &smem, &mask_rows)) {
    // with a workspace: the staged form (fp16 operand images and the rows'
    // bitmasks made once per call, the images copied in by one thread), its
    // tiles' blocks split over several CTAs where the tiles alone leave SMs
    // idle; without: the converting form, unsplit
    void* stage = nullptr;
    int ns = 1;
    float* part = nullptr;
    if (workspace != nullptr) {
      st = prefill_splits(S, p.G, Hkv, num_splits, &ns);
      if (st != I8KV_OK) return st;
      if (workspace_bytes < prefill_ws_bytes(S, Hq, Hkv, D, N, ns)) return I8KV_EWORKSPACE;
      stage = workspace;
      if (ns > 1)
        part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        (i8kv::prefill_stage_bytes(N, Hkv, D, S) + 255) / 256 * 256);
    } else if (num_splits > 1) {
      return I8KV_EWORKSPACE;  // the partials need one
    }
    cudaError_t e = i8kv::launch_dsa_prefill_tc(p, D, smem, mask_rows, stage, ns, part,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? I8KV_OK : cuda_fail(e);
  }
  return run(make_key(Path::kDsa, D, p.G, I8KV_CACHE_INT8, false), p,
             static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

i8kv_status paged_common(const uint16_t* q, const void* k_cache, const void* v_cache,
                         int32_t cache_dtype, const float* k_scale, const float* v_scale,
                         int32_t scale_kind, const int32_t* block_table,
                         const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t block_size, int32_t max_blocks, int64_t num_blocks,
                         float softmax_scale, const float* head_sink, float softcap,
                         int32_t window, int32_t num_splits, int32_t chunk, void* workspace,
                         size_t workspace_bytes, uint16_t* out, float* lse, int32_t* slots_out,
                         uint32_t* flags, void* stream) {
  if (B < 0 || max_blocks < 0 || num_blocks < 0 || block_size < 1 || num_splits < 0)
    return I8KV_EINVAL;
  if (!(softcap >= 0.f) || !std::isfinite(softcap) || window < -1) return I8KV_EINVAL;
  i8kv_status st = check_heads(Hq, Hkv, D);
  if (st != I8KV_OK) return st;
  if (block_size % 16 != 0) return I8KV_EUNSUPPORTED;
  if ((st = check_sigma(softmax_scale)) != I8KV_OK) return st;
  if (cache_dtype != I8KV_CACHE_INT8 && cache_dtype != I8KV_CACHE_FP16 &&
      cache_dtype != I8KV_CACHE_FP8)
    return I8KV_EINVAL;
  const bool fp16c = cache_dtype == I8KV_CACHE_FP16;
  if (!fp16c && (st = check_scales(k_scale, v_scale, scale_kind)) != I8KV_OK) return st;
  if (B > 0 && (q == nullptr || k_cache == nullptr || v_cache == nullptr ||
                seq_lens == nullptr || (max_blocks > 0 && block_table == nullptr)))
    return I8KV_EINVAL;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return I8KV_EALIGN;
  if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(lse, 4) ||
      !aligned(head_sink, 4) || !aligned(slots_out, 4) || !aligned(flags, 4))
    return I8KV_EALIGN;
  const int64_t cap = static_cast<int64_t>(max_blocks) * block_size;
  if (cap > INT32_MAX) return I8KV_EUNSUPPORTED;
  const int32_t G = Hq / Hkv;
  const KernelKey key = make_key(Path::kPaged, D, G, cache_dtype, true);
  const int64_t span = I8KV_WINDOW_SPAN(cap, window);
  if (num_splits == 0) {
    st = plan(key, span, std::max(1, B * Hkv), I8KV_GEOM_WAVE, 0, &num_splits, &chunk, nullptr);
    if (st != I8KV_OK) return st;
  }
  // chunk 0 with num_splits > 1: balanced pieces cut on the device (at most
  // num_splits per row)
  const bool balanced = num_splits > 1 && chunk == 0;
  if (balanced) {
    if (num_splits > I8KV_MAX_SPLITS) return I8KV_EINVAL;
    if (slots_out != nullptr || B > i8kv::kLptMaxRows) return I8KV_EUNSUPPORTED;
  } else if ((st = check_geometry(span, num_splits, chunk, window >= 0 ? cap : 0)) != I8KV_OK) {
    return st;
  }
  DecodeParams p{};
  if ((st = set_workspace(p, workspace, workspace_bytes, B * Hkv, num_splits, G, D)) != I8KV_OK)
    return st;
  if (out == nullptr && num_splits == 1 && B > 0) return I8KV_EINVAL;  // nowhere to write
  if (B == 0) return I8KV_OK;
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.k_scale = fp16c ? nullptr : k_scale;
  p.v_scale = fp16c ? nullptr : v_scale;
  p.per_channel = scale_kind == I8KV_SCALE_PER_CHANNEL;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.sink = head_sink;
  p.out = out;
  p.lse = lse;
  p.slots_out = slots_out;
  p.flags = flags;
  p.cache_rows = num_blocks;
  p.rows = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.bs = block_size;
  p.bs_log2 = -1;
  for (int sh = 4; sh < 31; ++sh)
    if (block_size == (1 << sh)) p.bs_log2 = sh;
  p.max_blocks = max_blocks;
  p.num_splits = num_splits;
  p.chunk = chunk;
  p.sigma = softmax_scale;
  p.softcap = softcap;
  p.window = window;
  // longest-first dispatch: ragged batches of long chunks (a property of the
  // geometry, so eager and captured launches make the same choice)
  p.lpt = !balanced && B <= i8kv::kLptMaxRows && chunk >= i8kv::kLptMinChunk;
  if (balanced) {
    // about one wave of CTAs over the KV heads, at least one piece per row,
    // at most what the grid of ceil(num_splits / 2) CTAs per unit holds
    WaveInfo w{0, 0};
    if ((st = wave_of(key, &w)) != I8KV_OK) return st;
    p.balanced = 1;
    p.bal_round = w.round;
    p.bal_pieces = std::min<int32_t>(std::max<int32_t>(w.wave / Hkv, B),
                                     B * ((num_splits + 1) / 2));
  }
  return run(key, p, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

i8kv_status paged_decode(const uint16_t* q, const void* k_cache, const void* v_cache,
                         int32_t cache_dtype, const float* k_scale, const float* v_scale,
                         int32_t scale_kind, const int32_t* block_table,
                         const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t block_size, int32_t max_blocks, int64_t num_blocks,
                         float softmax_scale, const float* head_sink, int32_t num_splits,
                         int32_t chunk, void* workspace, size_t workspace_bytes, uint16_t* out,
                         float* lse, int32_t* slots_out, uint32_t* flags, void* stream) {
  return paged_common(q, k_cache, v_cache, cache_dtype, k_scale, v_scale, scale_kind, block_table,
                      seq_lens, B, Hq, Hkv, D, block_size, max_blocks, num_blocks, softmax_scale,
                      head_sink, 0.f, -1, num_splits, chunk, workspace, workspace_bytes, out, lse,
                      slots_out, flags, stream);
}

i8kv_status paged_decode_ex(const uint16_t* q, const void* k_cache, const void* v_cache,
                            int32_t cache_dtype, const float* k_scale, const float* v_scale,
                            int32_t scale_kind, const int32_t* block_table,
                            const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv,
                            int32_t D, int32_t block_size, int32_t max_blocks, int64_t num_blocks,
                            float softmax_scale, const float* head_sink, float softcap,
                            int32_t window, int32_t num_splits, int32_t chunk, void* workspace,
                            size_t workspace_bytes, uint16_t* out, float* lse,
                            int32_t* slots_out, uint32_t* flags, void* stream) {
  return paged_common(q, k_cache, v_cache, cache_dtype, k_scale, v_scale, scale_kind, block_table,
                      seq_lens, B, Hq, Hkv, D, block_size, max_blocks, num_blocks, softmax_scale,
                      head_sink, softcap, window, num_splits, chunk, workspace, workspace_bytes,
                      out, lse, slots_out, flags, stream);
}

i8kv_status split_combine(const float* acc, const float* m, const float* l, int32_t units,
                          int32_t num_splits, int32_t Hq, int32_t Hkv, int32_t D,
                          const float* head_sink, uint16_t* out, float* lse, void* stream) {
  if (units < 0 || num_splits < 1 || num_splits > I8KV_MAX_SPLITS) return I8KV_EINVAL;
  i8kv_status st = check_heads(Hq, Hkv, D);
  if (st != I8KV_OK) return st;
  if (units > 0 && (acc == nullptr || m == nullptr || l == nullptr || out == nullptr))
    return I8KV_EINVAL;
  if (!aligned(acc, 16) || !aligned(out, 16) || !aligned(m, 4) || !aligned(l, 4) ||
      !aligned(lse, 4) || !aligned(head_sink, 4))
    return I8KV_EALIGN;
  if (units == 0) return I8KV_OK;
  cudaError_t e = i8kv::launch_combine(acc, m, l, units, num_splits, Hq, Hkv, D, head_sink, out,
                                       lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? I8KV_OK : cuda_fail(e);
}

i8kv_status reshape_and_cache(const uint16_t* k_new, const uint16_t* v_new,
                              const int32_t* slot_mapping, int32_t num_tokens, int32_t Hkv,
                              int32_t D, void* k_cache, void* v_cache, int64_t num_slots,
                              const float* k_scale, const float* v_scale, int32_t scale_kind,
                              int32_t cache_dtype, uint32_t* flags, void* stream) {
  if (num_tokens < 0 || Hkv < 1 || D < 8 || num_slots < 0) return I8KV_EINVAL;
  if (cache_dtype != I8KV_CACHE_INT8 && cache_dtype != I8KV_CACHE_FP8) return I8KV_EINVAL;
  if (D % 8 != 0) return I8KV_EUNSUPPORTED;
  i8kv_status st = check_scales(k_scale, v_scale, scale_kind);
  if (st != I8KV_OK) return st;
  if (num_tokens > 0 && (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr ||
                         k_cache == nullptr || v_cache == nullptr))
    return I8KV_EINVAL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(slot_mapping, 4) || !aligned(flags, 4))
    return I8KV_EALIGN;
  if (num_tokens == 0) return I8KV_OK;
  cudaError_t e = i8kv::launch_reshape_and_cache(
      k_new, v_new, slot_mapping, num_tokens, Hkv, D, k_cache, v_cache, num_slots, k_scale, v_scale,
      scale_kind == I8KV_SCALE_PER_CHANNEL, cache_dtype == I8KV_CACHE_FP8, flags,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? I8KV_OK : cuda_fail(e);
}

i8kv_status fp8_to_fp16(const uint8_t* in, uint16_t* out, int64_t n, void* stream) {
  if (n < 0 || n % 4 != 0) return I8KV_EINVAL;
  if (n > 0 && (in == nullptr || out == nullptr)) return I8KV_EINVAL;
  if (!aligned(in, 16) || !aligned(out, 16)) return I8KV_EALIGN;
  cudaError_t e = i8kv::launch_fp8_to_fp16(in, out, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? I8KV_OK : cuda_fail(e);
}

i8kv_status int8_to_fp16(const int8_t* in, uint16_t* out, int64_t n, void* stream) {
  if (n < 0 || n % 4 != 0) return I8KV_EINVAL;
  if (n > 0 && (in == nullptr || out == nullptr)) return I8KV_EINVAL;
  if (!aligned(in, 16) || !aligned(out, 16)) return I8KV_EALIGN;
  cudaError_t e = i8kv::launch_int8_to_fp16(in, out, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? I8KV_OK : cuda_fail(e);
}

}  // extern "C"
