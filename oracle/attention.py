"""FP64 CPU oracle for split-KV GQA attention over an INT8 (or FP16) KV cache.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain reference that the
CUDA path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import it; the product package
``int8_kv_cache_gb300`` never does, and this module imports nothing from it.

What is computed (all in float64, from the inputs exactly as a kernel receives
them: fp16 queries, int8 codes, fp32 scales):

1. Dequantisation.  ``x = scale * code`` with a per-tensor scale (one number)
   or a per-channel scale indexed by (kv_head, channel).  An fp16 cache is
   taken as is.  [onnxruntime PR 29912 "PagedAttention: quantized KV cache ...",
   Schema (k_quant_type / v_quant_type = PER_TENSOR | PER_CHANNEL, k_scale /
   v_scale) and CUDA kernels ("all read paths dequantize with k_scale/v_scale").]
2. Gather.  Sparse candidates: the entries of a row's index list that lie in
   [0, N), in list order, duplicates kept; other entries are invalid and
   skipped [onnxruntime PR 33707, Summary of Changes §1 test sweep "x invalid
   indices"].  Paged: token t of sequence b sits in physical row
   ``block_table[b, t // bs] * bs + t % bs`` for t < min(seq_len, cap), with
   cap = max_blocks * bs [PR 29912, CUDA kernels: block-table-aware decode;
   capacity block_table.shape[1] * block_size].
3. GQA.  Query head h reads KV head h // G, G = Hq / Hkv (contiguous groups).
4. Softmax in the natural-log domain with max subtraction:
   s_t = sigma * sum_d Q[h,d] K[t,d];  m = max_t s_t;  Z = sum_t exp(s_t - m);
   O = sum_t exp(s_t - m) V_t / Z;  lse = m + ln Z
   [PR 33707 §1: scores and running maximum stay in natural-log units; the
   expected output is an FP64 reference with max-subtracted weights].
5. Head sink (optional, one logit per query head, same units as the scaled
   scores, no value row):  O <- O / (1 + exp(s_h - lse))  [PR 29912, CUDA
   kernels, ApplyHeadSink: exact post-hoc LSE rescale].  The returned lse is
   that of the attended candidates, without the sink.
6. Split form.  Positions are partitioned into chunks; each chunk publishes an
   un-normalised partial (m_k, l_k, a_k) with a_k = sum exp(s_t - m_k) V_t; an
   empty chunk publishes (-inf, 0, 0).  The combine is
   M = max m_k;  L = sum l_k e^(m_k - M);  O = sum a_k e^(m_k - M) / L;
   lse = M + ln L, then the sink [PR 33707 §2: every CTA of the split-K decode
   writes an un-normalized partial (running maximum, running sum, accumulator)
   and a merge kernel combines them].

An empty candidate set gives O = 0 and lse = -inf (reading: the pages do not
say; a split with no tiles publishes an empty partial [PR 33707 §2 tests], and
the whole-row case is taken the same way).

7. Paged-decode variants [PR 29912, CUDA kernels: the paged decode kernel has
   native head-sink, softcap, sliding-window and on-the-fly dequantisation].
   The pages name both options without defining them; the readings taken are
   the usual ones of that runtime's attention operators:
   - softcap c > 0: every scaled score s becomes c * tanh(s / c) before the
     softmax (c = 0: off).  The sink logit is not capped.
   - sliding window w >= 0: the decode query sits at position L - 1 (L the
     live length) and attends positions [max(0, L - 1 - w), L), i.e. itself
     and the w positions before it (w = -1: off).
   In the split form with a window, chunks are counted from the window start
   rounded down to a multiple of 16 tokens (the tile granule, so that no tile
   straddles a block), and the split geometry is taken over the span
   min(cap, w + 16) instead of cap; both depend on w only, never on L.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

SCALE_PER_TENSOR = 1
SCALE_PER_CHANNEL = 2


# --------------------------------------------------------------------------
# 1. dequantisation
# --------------------------------------------------------------------------

def e4m3fn_value(code: int) -> float:
    """Value of one float8 e4m3fn bit pattern (OCP 8-bit floating point, E4M3:
    sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is
    subnormal, m * 2^-9; S.1111.111 is NaN; there are no infinities)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3FN_TABLE = np.array([e4m3fn_value(c) for c in range(256)], dtype=np.float64)


def dequantize(codes: np.ndarray, scale: np.ndarray, scale_kind: int, kv_head: int) -> np.ndarray:
    """Rows ``codes[..., D]`` of one KV head -> float64 values.

    per-tensor: scale[0] * code;  per-channel: scale[kv_head, d] * code.
    An int8 array holds INT8 codes, a uint8 array float8 e4m3fn bit patterns
    (whose values the scales multiply the same way) [PR 29912, Schema: the
    cache element type is one of float16, bfloat16, int8, float8e4m3fn].
    A float16 cache is returned as is (no scale).
    """
    codes = np.asarray(codes)
    if codes.dtype == np.uint8:
        x = _E4M3FN_TABLE[codes]
    else:
        x = codes.astype(np.float64)
    if codes.dtype == np.float16:
        return x
    if scale_kind == SCALE_PER_TENSOR:
        return x * float(np.asarray(scale, dtype=np.float64).reshape(-1)[0])
    if scale_kind == SCALE_PER_CHANNEL:
        return x * np.asarray(scale, dtype=np.float64)[kv_head]
    raise ValueError(f"unknown scale kind {scale_kind}")


# --------------------------------------------------------------------------
# 4./5. one query head against a candidate set
# --------------------------------------------------------------------------

def scores(q: np.ndarray, K: np.ndarray, sigma: float, softcap: float = 0.0) -> np.ndarray:
    """s_t = sigma * <q, K_t>, then c * tanh(s_t / c) when softcap c > 0."""
    s = sigma * (K @ np.asarray(q, dtype=np.float64))
    if softcap > 0.0:
        s = softcap * np.tanh(s / softcap)
    return s


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, sigma: float,
           softcap: float = 0.0) -> Tuple[np.ndarray, float]:
    """Softmax attention of one query vector ``q[D]`` over rows ``K[T, D]``,
    ``V[T, D]`` (float64).  Returns (O[D], lse)."""
    q = np.asarray(q, dtype=np.float64)
    T = K.shape[0]
    if T == 0:
        return np.zeros(V.shape[1], dtype=np.float64), -math.inf
    s = scores(q, K, sigma, softcap)
    m = float(np.max(s))
    w = np.exp(s - m)
    Z = float(np.sum(w))
    o = (w @ V) / Z
    return o, m + math.log(Z)


def apply_head_sink(o: np.ndarray, lse: float, s_h: Optional[float]) -> np.ndarray:
    """O <- O / (1 + exp(s_h - lse)); no sink leaves O unchanged.  With an empty
    candidate set (lse = -inf) O is already zero and stays zero."""
    if s_h is None or lse == -math.inf:
        return o
    return o / (1.0 + math.exp(float(s_h) - lse))


def _sink_of(sink, h):
    return None if sink is None else float(np.asarray(sink, dtype=np.float64)[h])


# --------------------------------------------------------------------------
# 2. gathers
# --------------------------------------------------------------------------

def sparse_candidates(idx_row: np.ndarray, N: int) -> np.ndarray:
    """Valid entries of one candidate list, in list order, duplicates kept."""
    r = np.asarray(idx_row, dtype=np.int64)
    return r[(r >= 0) & (r < N)]


def paged_slots(block_table: np.ndarray, seq_lens: np.ndarray, bs: int,
                window: int = -1) -> np.ndarray:
    """Physical row of every attended token position: ``out[b, t] =
    bt[b, t//bs]*bs + t%bs`` for window_start <= t < min(seq_len_b, cap), else
    -1.  Shape [B, cap], int64."""
    bt = np.asarray(block_table, dtype=np.int64)
    B, mb = bt.shape
    cap = mb * bs
    out = np.full((B, cap), -1, dtype=np.int64)
    for b in range(B):
        L = live_length(int(seq_lens[b]), cap)
        for t in range(window_start(L, window), L):
            out[b, t] = bt[b, t // bs] * bs + t % bs
    return out


def window_start(L: int, window: int) -> int:
    """First attended position of a decode query at position L - 1: L - 1 - w
    (not below 0) with a window w >= 0, else 0."""
    return max(0, L - 1 - window) if window >= 0 else 0


def window_span(cap: int, window: int) -> int:
    """Positions the splits of a windowed decode must cover: the window's w + 1
    positions plus up to 15 before its start (chunks start 16-aligned)."""
    return min(cap, window + 16) if window >= 0 else cap


def live_length(seq_len: int, cap: int) -> int:
    """A sequence's attended length: its seq_len clamped to [0, cap]."""
    return max(0, min(int(seq_len), int(cap)))


# --------------------------------------------------------------------------
# whole-row references
# --------------------------------------------------------------------------

def sparse_attention(q, k_codes, v_codes, k_scale, v_scale, scale_kind, idx, sigma, sink=None):
    """Sparse-candidate attention (decode rows or prefill rows alike).

    q [S, Hq, D] fp16; caches [N, Hkv, D]; idx [S, max_sel].
    Returns O [S, Hq, D] float64 and lse [S, Hq] float64.
    """
    S, Hq, D = q.shape
    N, Hkv, _ = k_codes.shape
    G = Hq // Hkv
    O = np.zeros((S, Hq, D), dtype=np.float64)
    L = np.full((S, Hq), -math.inf, dtype=np.float64)
    for r in range(S):
        rows = sparse_candidates(idx[r], N)
        for g in range(Hkv):
            K = dequantize(k_codes[rows, g, :], k_scale, scale_kind, g)
            V = dequantize(v_codes[rows, g, :], v_scale, scale_kind, g)
            for h in range(g * G, (g + 1) * G):
                o, lse = attend(q[r, h].astype(np.float64), K, V, sigma)
                O[r, h] = apply_head_sink(o, lse, _sink_of(sink, h))
                L[r, h] = lse
    return O, L


def paged_attention(q, k_cache, v_cache, k_scale, v_scale, scale_kind, block_table, seq_lens,
                    sigma, sink=None, softcap: float = 0.0, window: int = -1):
    """Paged-cache decode: one query row per sequence.

    q [B, Hq, D]; caches [num_blocks, bs, Hkv, D]; block_table [B, max_blocks].
    Returns O [B, Hq, D], lse [B, Hq] (float64).
    """
    B, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    G = Hq // Hkv
    kf = k_cache.reshape(nb * bs, Hkv, D)
    vf = v_cache.reshape(nb * bs, Hkv, D)
    slots = paged_slots(block_table, seq_lens, bs, window)
    O = np.zeros((B, Hq, D), dtype=np.float64)
    L = np.full((B, Hq), -math.inf, dtype=np.float64)
    for b in range(B):
        rows = slots[b][slots[b] >= 0]
        for g in range(Hkv):
            K = dequantize(kf[rows, g, :], k_scale, scale_kind, g)
            V = dequantize(vf[rows, g, :], v_scale, scale_kind, g)
            for h in range(g * G, (g + 1) * G):
                o, lse = attend(q[b, h].astype(np.float64), K, V, sigma, softcap)
                O[b, h] = apply_head_sink(o, lse, _sink_of(sink, h))
                L[b, h] = lse
    return O, L


# --------------------------------------------------------------------------
# 6. split form: partials and the log-sum-exp combine
# --------------------------------------------------------------------------

def partial(q: np.ndarray, K: np.ndarray, V: np.ndarray, sigma: float, softcap: float = 0.0):
    """Un-normalised partial of one chunk: (m, l, a) with a = sum e^(s-m) V.
    An empty chunk gives (-inf, 0, 0)."""
    D = V.shape[1]
    if K.shape[0] == 0:
        return -math.inf, 0.0, np.zeros(D, dtype=np.float64)
    s = scores(q, K, sigma, softcap)
    m = float(np.max(s))
    w = np.exp(s - m)
    return m, float(np.sum(w)), w @ V


def combine(ms: Sequence[float], ls: Sequence[float], accs: Sequence[np.ndarray],
            s_h: Optional[float] = None) -> Tuple[np.ndarray, float]:
    """Log-sum-exp merge of split partials, then the head sink."""
    ms = np.asarray(ms, dtype=np.float64)
    D = len(accs[0]) if len(accs) else 0
    live = np.isfinite(ms)
    if not np.any(live):
        return np.zeros(D, dtype=np.float64), -math.inf
    M = float(np.max(ms[live]))
    f = np.where(live, np.exp(np.where(live, ms - M, 0.0)), 0.0)
    Lsum = float(np.sum(f * np.asarray(ls, dtype=np.float64)))
    o = np.zeros(D, dtype=np.float64)
    for k in range(len(accs)):
        if live[k]:
            o += f[k] * np.asarray(accs[k], dtype=np.float64)
    o /= Lsum
    lse = M + math.log(Lsum)
    return apply_head_sink(o, lse, s_h), lse


def chunk_bounds(length: int, chunk: int, num_splits: int) -> List[Tuple[int, int]]:
    """Split k covers positions [k*chunk, (k+1)*chunk) intersected with [0, length)."""
    out = []
    for k in range(num_splits):
        lo = min(k * chunk, length)
        hi = min((k + 1) * chunk, length)
        out.append((lo, hi))
    return out


def sparse_split_partials(q, k_codes, v_codes, k_scale, v_scale, scale_kind, idx, sigma,
                          num_splits: int, chunk: int):
    """Partials of the split form over list positions: split k of row r covers
    list positions [k*chunk, (k+1)*chunk) of idx[r] (invalid entries skipped).

    Returns m, l [S, Hq, splits] and acc [S, Hq, splits, D] (float64)."""
    S, Hq, D = q.shape
    N, Hkv, _ = k_codes.shape
    G = Hq // Hkv
    m = np.full((S, Hq, num_splits), -math.inf)
    l = np.zeros((S, Hq, num_splits))
    a = np.zeros((S, Hq, num_splits, D))
    max_sel = idx.shape[1]
    for r in range(S):
        for k, (lo, hi) in enumerate(chunk_bounds(max_sel, chunk, num_splits)):
            rows = sparse_candidates(idx[r, lo:hi], N)
            for g in range(Hkv):
                K = dequantize(k_codes[rows, g, :], k_scale, scale_kind, g)
                V = dequantize(v_codes[rows, g, :], v_scale, scale_kind, g)
                for h in range(g * G, (g + 1) * G):
                    m[r, h, k], l[r, h, k], a[r, h, k] = partial(q[r, h], K, V, sigma)
    return m, l, a


def prefill_block_ranges(idx, N: int, G: int, num_splits: int, tile: int = 128,
                         block: int = 128) -> List[List[Tuple[int, int]]]:
    """Position ranges of the split tensor-core prefill (reading 13 of the
    design: the pages' prefill has no splits; this is the split-K partial and
    merge of PR 33707 §2 applied to a tile's blocks).  Query vectors r*G + j
    of one KV head form tiles of `tile` consecutive vectors; a tile's blocks
    are the `block`-position blocks holding a valid candidate of any of its
    rows, ranked in position order; split k takes ranks
    [k*cnt // num_splits, (k+1)*cnt // num_splits) and the positions from its
    first block to the next split's first block (split 0 from 0, the last split
    to N; a rank past the last block stands for the block after the tile's
    last one).  Returns, per tile, the num_splits (lo, hi) ranges."""
    S = idx.shape[0]
    nvec = S * G
    out = []
    for t in range(-(-nvec // tile)):
        r_lo = (t * tile) // G
        r_hi = (min(t * tile + tile - 1, nvec - 1)) // G
        pos = np.concatenate([sparse_candidates(idx[r], N) for r in range(r_lo, r_hi + 1)])
        blocks = sorted(set((pos // block).tolist()))
        cnt = len(blocks)
        past = (blocks[-1] + 1) if cnt else 0
        first = lambda rank: blocks[rank] if rank < cnt else past  # noqa: E731
        ranges = []
        for k in range(num_splits):
            r0, r1 = k * cnt // num_splits, (k + 1) * cnt // num_splits
            lo = 0 if k == 0 else first(r0) * block
            hi = N if k == num_splits - 1 else first(r1) * block
            ranges.append((lo, hi))
        out.append(ranges)
    return out


def prefill_split_partials(q, k_codes, v_codes, k_scale, v_scale, scale_kind, idx, sigma,
                           num_splits: int, tile: int = 128, block: int = 128):
    """Partials of the split tensor-core prefill: vector (r, h) of KV head g
    lies in tile (r*G + h - g*G) // tile of that head, and its split k covers
    the candidates of row r at the positions of that tile's range k
    (prefill_block_ranges).  Returns m, l [S, Hq, splits] and acc
    [S, Hq, splits, D] (float64)."""
    S, Hq, D = q.shape
    N, Hkv, _ = k_codes.shape
    G = Hq // Hkv
    ranges = prefill_block_ranges(idx, N, G, num_splits, tile, block)
    m = np.full((S, Hq, num_splits), -math.inf)
    l = np.zeros((S, Hq, num_splits))
    a = np.zeros((S, Hq, num_splits, D))
    for r in range(S):
        cand = sparse_candidates(idx[r], N)
        for j in range(G):
            t = (r * G + j) // tile
            for k, (lo, hi) in enumerate(ranges[t]):
                rows = cand[(cand >= lo) & (cand < hi)]
                for g in range(Hkv):
                    K = dequantize(k_codes[rows, g, :], k_scale, scale_kind, g)
                    V = dequantize(v_codes[rows, g, :], v_scale, scale_kind, g)
                    h = g * G + j
                    m[r, h, k], l[r, h, k], a[r, h, k] = partial(q[r, h], K, V, sigma)
    return m, l, a


def window_chunk_bounds(L: int, window: int, chunk: int,
                        num_splits: int) -> List[Tuple[int, int]]:
    """Split k of a windowed row covers [b16 + k*chunk, b16 + (k+1)*chunk)
    intersected with [start, L), where start = window_start(L, window) and b16
    is start rounded down to a multiple of 16."""
    start = window_start(L, window)
    b16 = start - start % 16
    out = []
    for k in range(num_splits):
        lo = max(start, min(b16 + k * chunk, L))
        hi = max(lo, min(b16 + (k + 1) * chunk, L))
        out.append((lo, hi))
    return out


def paged_split_partials(q, k_cache, v_cache, k_scale, v_scale, scale_kind, block_table,
                         seq_lens, sigma, num_splits: int, chunk: int, softcap: float = 0.0,
                         window: int = -1):
    """Partials of the split form over token positions of each sequence
    (chunks from position 0, or from the window start as in
    ``window_chunk_bounds``)."""
    B, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    G = Hq // Hkv
    kf = k_cache.reshape(nb * bs, Hkv, D)
    vf = v_cache.reshape(nb * bs, Hkv, D)
    slots = paged_slots(block_table, seq_lens, bs)
    cap = slots.shape[1]
    m = np.full((B, Hq, num_splits), -math.inf)
    l = np.zeros((B, Hq, num_splits))
    a = np.zeros((B, Hq, num_splits, D))
    for b in range(B):
        Lb = live_length(int(seq_lens[b]), cap)
        bounds = (window_chunk_bounds(Lb, window, chunk, num_splits) if window >= 0
                  else chunk_bounds(Lb, chunk, num_splits))
        for k, (lo, hi) in enumerate(bounds):
            rows = slots[b, lo:hi]
            for g in range(Hkv):
                K = dequantize(kf[rows, g, :], k_scale, scale_kind, g)
                V = dequantize(vf[rows, g, :], v_scale, scale_kind, g)
                for h in range(g * G, (g + 1) * G):
                    m[b, h, k], l[b, h, k], a[b, h, k] = partial(q[b, h], K, V, sigma,
                                                                 softcap)
    return m, l, a


def combine_all(m, l, a, sink=None):
    """Combine partials [R, Hq, splits(, D)] row by row -> O [R, Hq, D], lse [R, Hq]."""
    R, Hq, ns = m.shape
    D = a.shape[-1]
    O = np.zeros((R, Hq, D))
    L = np.full((R, Hq), -math.inf)
    for r in range(R):
        for h in range(Hq):
            O[r, h], L[r, h] = combine(m[r, h], l[r, h], list(a[r, h]), _sink_of(sink, h))
    return O, L
