"""Seeded synthetic inputs for the INT8 KV-cache decode / prefill path.

This module only *draws* inputs: queries, caches (as int8 codes plus the fp32
scales that produced them), candidate index lists, block tables, lengths and
head-sink logits.  It contains none of the attention arithmetic (no gather,
dequantisation, softmax, split or combine).  Both the FP64 oracle's tests and
the CUDA path's tests / benchmark use these generators, so that the two sides
see byte-identical inputs; nothing else is shared between them.

Every generator takes a ``seed`` and uses ``numpy.random.Generator(PCG64(seed))``
and draws in a fixed order: Q, K, V, (scales are derived), indices or block
table, sinks.

The shapes and distributions follow the workloads the pages measure:

* tiny decode: 1 sequence, 4 query / 1 KV head, head_dim 64, 128 tokens;
* sparse-candidate decode (onnxruntime PR 33707, "Performance": 24 query /
  2 KV heads, head size 256, 2048 selected candidates, scale 1/16);
* paged decode (onnxruntime PR 29912, "Paged decode kernel": block-table
  layout, per-channel INT8 scales, head sink);
* deep-context split sweep (onnx-genai PR 1350, "Summary": 16 decode rows,
  ~2600-token context within cap 4096);
* sparse-candidate prefill (onnxruntime PR 33707, "Performance", prefill
  table: 2048 rows, context 8192, 2048 selected).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

SCALE_PER_TENSOR = 1
SCALE_PER_CHANNEL = 2


def make_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def quantize_int8(x: np.ndarray, scale_kind: int):
    """Synthesise an INT8 cache from fp32 values ``x[..., Hkv, D]``.

    Symmetric codes in [-127, 127] with ``scale = amax / 127`` taken over all
    tokens, per (kv_head, channel) for per-channel scales or over the whole
    tensor for a per-tensor scale; an all-zero channel gets scale 1.  Codes are
    ``clip(rint(x / scale))`` (round half to even).  This is how the test data
    are made, not a step of the decode path.
    """
    x = np.asarray(x, dtype=np.float32)
    lead = tuple(range(x.ndim - 2))
    if scale_kind == SCALE_PER_CHANNEL:
        amax = np.abs(x).max(axis=lead)  # [Hkv, D]
    elif scale_kind == SCALE_PER_TENSOR:
        amax = np.abs(x).max().reshape(1)
    else:
        raise ValueError(f"unknown scale kind {scale_kind}")
    scale = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    if scale_kind == SCALE_PER_TENSOR:
        codes = np.rint(x / scale[0])
    else:
        codes = np.rint(x / scale)
    codes = np.clip(codes, -127, 127).astype(np.int8)
    return codes, scale


def quantize_fp8(x: np.ndarray, scale_kind: int):
    """Synthesise a float8 e4m3fn cache (uint8 bit patterns) from fp32 values
    ``x[..., Hkv, D]``: ``scale = amax / 448`` (the largest finite e4m3fn
    value) per (kv_head, channel) or per tensor, values ``x / scale`` converted
    by PyTorch's float8_e4m3fn dtype (round to nearest even).  Test data only."""
    import torch
    x = np.asarray(x, dtype=np.float32)
    lead = tuple(range(x.ndim - 2))
    if scale_kind == SCALE_PER_CHANNEL:
        amax = np.abs(x).max(axis=lead)
    elif scale_kind == SCALE_PER_TENSOR:
        amax = np.abs(x).max().reshape(1)
    else:
        raise ValueError(f"unknown scale kind {scale_kind}")
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    y = x / (scale[0] if scale_kind == SCALE_PER_TENSOR else scale)
    y = np.clip(y, -448.0, 448.0).astype(np.float32)
    codes = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy().copy(), scale


@dataclass
class SparseCase:
    """Inputs of a sparse-candidate (DSA) call: each query row has its own list."""

    q: np.ndarray  # [S, Hq, D] float16
    k_codes: np.ndarray  # [N, Hkv, D] int8
    v_codes: np.ndarray  # [N, Hkv, D] int8
    k_scale: np.ndarray  # [1] or [Hkv, D] float32
    v_scale: np.ndarray  # [1] or [Hkv, D] float32
    scale_kind: int
    idx: np.ndarray  # [S, max_sel] int32, entries <0 or >=N are invalid
    sigma: float
    sink: Optional[np.ndarray] = None  # [Hq] float32
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        S, Hq, D = self.q.shape
        return dict(S=S, Hq=Hq, Hkv=self.k_codes.shape[1], D=D, N=self.k_codes.shape[0],
                    max_sel=self.idx.shape[1])


@dataclass
class PagedCase:
    """Inputs of a paged-cache decode call (one query row per sequence)."""

    q: np.ndarray  # [B, Hq, D] float16
    k_cache: np.ndarray  # [num_blocks, bs, Hkv, D] int8 or float16
    v_cache: np.ndarray
    k_scale: np.ndarray  # [1] or [Hkv, D] float32 (ignored for a float16 cache)
    v_scale: np.ndarray
    scale_kind: int
    block_table: np.ndarray  # [B, max_blocks] int32, unused entries -1
    seq_lens: np.ndarray  # [B] int32
    sigma: float
    sink: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, Hq, D = self.q.shape
        nb, bs, Hkv, _ = self.k_cache.shape
        return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, bs=bs, num_blocks=nb,
                    max_blocks=self.block_table.shape[1])


def _channel_std(rng, Hkv, D):
    # per-(kv_head, channel) standard deviation, log-uniform in [0.5, 2]
    return np.exp(rng.uniform(np.log(0.5), np.log(2.0), size=(Hkv, D))).astype(np.float32)


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def _sorted_unique(rng, hi_exclusive, n):
    return np.sort(rng.choice(hi_exclusive, size=n, replace=False)).astype(np.int32)


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

def tiny_decode(seed: int = 0, scale_kind: int = SCALE_PER_CHANNEL) -> PagedCase:
    """1 sequence, 1 query row, 4 query / 1 KV head, head_dim 64, 128 tokens
    (identity block table, block size 16), sigma = 1/sqrt(64)."""
    rng = make_rng(seed)
    Hq, Hkv, D, T, bs = 4, 1, 64, 128, 16
    q = _normal(rng, (1, Hq, D)).astype(np.float16)
    k = _normal(rng, (T, Hkv, D))
    v = _normal(rng, (T, Hkv, D))
    kc, ks = quantize_int8(k, scale_kind)
    vc, vs = quantize_int8(v, scale_kind)
    nb = T // bs
    return PagedCase(q=q, k_cache=kc.reshape(nb, bs, Hkv, D), v_cache=vc.reshape(nb, bs, Hkv, D),
                     k_scale=ks, v_scale=vs, scale_kind=scale_kind,
                     block_table=np.arange(nb, dtype=np.int32).reshape(1, nb),
                     seq_lens=np.array([T], dtype=np.int32), sigma=1.0 / 8.0, sink=None,
                     meta=dict(name="tiny decode"))


def sparse_decode(S: int, seed: int = 0, Hq: int = 24, Hkv: int = 2, D: int = 256,
                  N: int = 16384, n_sel: int = 2048, sink: bool = False) -> SparseCase:
    """Sparse-candidate INT8 decode: S rows, each with ``n_sel`` sorted unique
    candidates drawn uniformly from the ``N``-token cache; per-channel scales
    with channel std log-uniform in [0.5, 2]; sigma = 1/16."""
    rng = make_rng(seed)
    q = _normal(rng, (S, Hq, D)).astype(np.float16)
    std = _channel_std(rng, Hkv, D)
    k = _normal(rng, (N, Hkv, D)) * std
    v = _normal(rng, (N, Hkv, D)) * std
    kc, ks = quantize_int8(k, SCALE_PER_CHANNEL)
    vc, vs = quantize_int8(v, SCALE_PER_CHANNEL)
    idx = np.stack([_sorted_unique(rng, N, n_sel) for _ in range(S)]) if S > 0 else \
        np.zeros((0, n_sel), np.int32)
    snk = _normal(rng, (Hq,)) if sink else None
    return SparseCase(q=q, k_codes=kc, v_codes=vc, k_scale=ks, v_scale=vs,
                      scale_kind=SCALE_PER_CHANNEL, idx=idx, sigma=1.0 / 16.0, sink=snk,
                      meta=dict(name=f"sparse decode S={S}"))


def paged_decode(seed: int = 0, B: int = 16, len_lo: int = 512, len_hi: int = 8192,
                 bs: int = 16, max_blocks: int = 512, Hq: int = 32, Hkv: int = 8, D: int = 128,
                 scale_kind: int = SCALE_PER_CHANNEL, sink: bool = True,
                 cache: str = "int8") -> PagedCase:
    """Paged INT8 (or float8 e4m3fn) decode: lengths uniform in [len_lo,
    len_hi]; the physical pool holds exactly sum(ceil(len/bs)) blocks and the
    block table is a random permutation of them (unused entries -1);
    sigma = 1/sqrt(D)."""
    rng = make_rng(seed)
    quant = quantize_fp8 if cache == "fp8" else quantize_int8
    lens = rng.integers(len_lo, len_hi + 1, size=B).astype(np.int32)
    nblk = (lens + bs - 1) // bs
    P = int(nblk.sum())
    q = _normal(rng, (B, Hq, D)).astype(np.float16)
    k = _normal(rng, (P, bs, Hkv, D))
    kc, ks = quant(k, scale_kind)
    del k
    v = _normal(rng, (P, bs, Hkv, D))
    vc, vs = quant(v, scale_kind)
    del v
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += nblk[b]
    snk = _normal(rng, (Hq,)) if sink else None
    return PagedCase(q=q, k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs, scale_kind=scale_kind,
                     block_table=bt, seq_lens=lens, sigma=1.0 / float(np.sqrt(D)), sink=snk,
                     meta=dict(name="paged decode"))


def deep_context(seed: int = 0, cache: str = "int8", B: int = 16, cap: int = 4096,
                 live: int = 2600, Hq: int = 16, Hkv: int = 2, D: int = 128, bs: int = 16,
                 sink: bool = False) -> PagedCase:
    """Deep-context split sweep: B sequences with their own contiguous cache of
    ``cap`` tokens (identity block table), live length ``live``; int8 or float8
    e4m3fn cache with per-channel scales, or a float16 cache; sigma = 1/sqrt(D)."""
    rng = make_rng(seed)
    mb = cap // bs
    q = _normal(rng, (B, Hq, D)).astype(np.float16)
    k = _normal(rng, (B * mb, bs, Hkv, D))
    v = _normal(rng, (B * mb, bs, Hkv, D))
    if cache == "int8":
        kc, ks = quantize_int8(k, SCALE_PER_CHANNEL)
        vc, vs = quantize_int8(v, SCALE_PER_CHANNEL)
    elif cache == "fp8":
        kc, ks = quantize_fp8(k, SCALE_PER_CHANNEL)
        vc, vs = quantize_fp8(v, SCALE_PER_CHANNEL)
    elif cache == "fp16":
        kc, vc = k.astype(np.float16), v.astype(np.float16)
        ks = vs = np.ones((Hkv, D), np.float32)
    else:
        raise ValueError(cache)
    bt = np.arange(B * mb, dtype=np.int32).reshape(B, mb)
    lens = np.full((B,), live, dtype=np.int32)
    snk = _normal(rng, (Hq,)) if sink else None
    return PagedCase(q=q, k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs,
                     scale_kind=SCALE_PER_CHANNEL, block_table=bt, seq_lens=lens,
                     sigma=1.0 / float(np.sqrt(D)), sink=snk,
                     meta=dict(name=f"deep context {cache}", cap=cap))


def sparse_prefill(seed: int = 0, rows: int = 2048, N: int = 8192, Hq: int = 24, Hkv: int = 2,
                   D: int = 256, n_sel: int = 2048, literal: bool = False,
                   row_subset: Optional[np.ndarray] = None) -> SparseCase:
    """Sparse-candidate prefill.  Row i sits at position p_i = N - rows + i (or
    p_i = i with ``literal``) and attends min(n_sel, p_i + 1) sorted unique
    candidates drawn uniformly from [0, p_i]; unused list slots are -1.
    ``row_subset`` keeps only the listed rows (same draws as the full case)."""
    rng = make_rng(seed)
    q = _normal(rng, (rows, Hq, D)).astype(np.float16)
    std = _channel_std(rng, Hkv, D)
    k = _normal(rng, (N, Hkv, D)) * std
    v = _normal(rng, (N, Hkv, D)) * std
    kc, ks = quantize_int8(k, SCALE_PER_CHANNEL)
    vc, vs = quantize_int8(v, SCALE_PER_CHANNEL)
    idx = np.full((rows, n_sel), -1, dtype=np.int32)
    for i in range(rows):
        p = i if literal else N - rows + i
        n = min(n_sel, p + 1)
        idx[i, :n] = _sorted_unique(rng, p + 1, n)
    if row_subset is not None:
        q, idx = q[row_subset], idx[row_subset]
    return SparseCase(q=q, k_codes=kc, v_codes=vc, k_scale=ks, v_scale=vs,
                      scale_kind=SCALE_PER_CHANNEL, idx=idx, sigma=1.0 / 16.0, sink=None,
                      meta=dict(name="sparse prefill" + (" (literal)" if literal else "")))


# --------------------------------------------------------------------------
# general random cases for the parity sweeps
# --------------------------------------------------------------------------

def random_sparse(seed: int, S: int, Hq: int, Hkv: int, D: int, N: int, max_sel: int,
                  n_valid: Optional[int] = None, invalid_frac: float = 0.0,
                  scale_kind: int = SCALE_PER_CHANNEL, sink: bool = False,
                  sigma: Optional[float] = None, q_std: float = 1.0,
                  sorted_lists: bool = False) -> SparseCase:
    """Random sparse case: each row's list has ``n_valid`` (default max_sel)
    entries drawn without replacement from [0, N); a fraction ``invalid_frac``
    of them is replaced by out-of-range values (-1, -7, N, N+5); slots past
    ``n_valid`` are -1."""
    rng = make_rng(seed)
    q = (_normal(rng, (S, Hq, D)) * np.float32(q_std)).astype(np.float16)
    std = _channel_std(rng, Hkv, D)
    k = _normal(rng, (N, Hkv, D)) * std
    v = _normal(rng, (N, Hkv, D)) * std
    kc, ks = quantize_int8(k, scale_kind)
    vc, vs = quantize_int8(v, scale_kind)
    nv = max_sel if n_valid is None else n_valid
    idx = np.full((S, max_sel), -1, dtype=np.int32)
    bad = np.array([-1, -7, N, N + 5], dtype=np.int64)
    for r in range(S):
        take = min(nv, N)
        sel = rng.choice(N, size=take, replace=False).astype(np.int64)
        if sorted_lists:
            sel = np.sort(sel)
        if invalid_frac > 0 and take > 0:
            mask = rng.random(take) < invalid_frac
            sel[mask] = bad[rng.integers(0, len(bad), size=int(mask.sum()))]
        idx[r, :take] = sel.astype(np.int32)
    snk = _normal(rng, (Hq,)) if sink else None
    sg = (1.0 / float(np.sqrt(D))) if sigma is None else sigma
    return SparseCase(q=q, k_codes=kc, v_codes=vc, k_scale=ks, v_scale=vs, scale_kind=scale_kind,
                      idx=idx, sigma=sg, sink=snk, meta=dict(name="random sparse"))


def random_paged(seed: int, B: int, Hq: int, Hkv: int, D: int, bs: int, max_blocks: int,
                 lens, scale_kind: int = SCALE_PER_CHANNEL, sink: bool = False,
                 cache: str = "int8", spare_blocks: int = 3) -> PagedCase:
    """Random paged case with explicit lengths (a length may exceed the cap
    max_blocks*bs; the table then only covers the cap).  The pool has a few
    spare blocks beyond those referenced and the table is a permutation."""
    rng = make_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    cap = max_blocks * bs
    nblk = np.minimum((np.maximum(lens, 0) + bs) // bs, max_blocks)  # room for one more token
    P = int(nblk.sum()) + spare_blocks
    q = _normal(rng, (B, Hq, D)).astype(np.float16)
    k = _normal(rng, (P, bs, Hkv, D))
    v = _normal(rng, (P, bs, Hkv, D))
    if cache == "int8":
        kc, ks = quantize_int8(k, scale_kind)
        vc, vs = quantize_int8(v, scale_kind)
    elif cache == "fp8":
        kc, ks = quantize_fp8(k, scale_kind)
        vc, vs = quantize_fp8(v, scale_kind)
    else:
        kc, vc = k.astype(np.float16), v.astype(np.float16)
        ks = vs = np.ones((Hkv, D), np.float32)
        scale_kind = SCALE_PER_CHANNEL
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += nblk[b]
    snk = _normal(rng, (Hq,)) if sink else None
    return PagedCase(q=q, k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs, scale_kind=scale_kind,
                     block_table=bt, seq_lens=lens, sigma=1.0 / float(np.sqrt(D)), sink=snk,
                     meta=dict(name="random paged", cap=cap))


# --------------------------------------------------------------------------
# two-candidate analytic constructions (an otherwise empty cache)
# --------------------------------------------------------------------------

def two_candidate(q_vec, kA, kB, vA, vB, k_scale: float, v_scale: float, sigma: float,
                  spread: bool = False, Hq: int = 4, Hkv: int = 1, N: int = 520,
                  rows_at=(17, 403)) -> SparseCase:
    """Two selected candidates of an otherwise all-zero INT8 cache, per-tensor
    scales.  Every query head gets the same query vector ``q_vec`` (exactly
    representable in fp16).  The list has 192 slots (three 64-candidate
    tiles); the two valid entries sit in slots 0 and 1, or, with ``spread``,
    in slots 0 and 191 (first and last tile); the other slots are -1."""
    q_vec = np.asarray(q_vec, dtype=np.float64)
    D = q_vec.shape[0]
    q16 = q_vec.astype(np.float16)
    if not np.array_equal(q16.astype(np.float64), q_vec):
        raise ValueError("query not exactly representable in fp16")
    kc = np.zeros((N, Hkv, D), np.int8)
    vc = np.zeros((N, Hkv, D), np.int8)
    a, b = rows_at
    for g in range(Hkv):
        kc[a, g], kc[b, g] = np.asarray(kA, np.int8), np.asarray(kB, np.int8)
        vc[a, g], vc[b, g] = np.asarray(vA, np.int8), np.asarray(vB, np.int8)
    idx = np.full((1, 192), -1, np.int32)
    idx[0, 0] = a
    idx[0, 191 if spread else 1] = b
    q = np.broadcast_to(q16, (1, Hq, D)).copy()
    return SparseCase(q=q, k_codes=kc, v_codes=vc,
                      k_scale=np.array([k_scale], np.float32), v_scale=np.array([v_scale], np.float32),
                      scale_kind=SCALE_PER_TENSOR, idx=idx, sigma=float(sigma), sink=None,
                      meta=dict(name="two candidates", spread=spread))


def signed_cancellation_case(D: int = 64, spread: bool = False) -> SparseCase:
    """Probabilities 0.5 +- 2^-14 on values +-4064 (codes +-127, value scale 32):
    logit gap ln((2^13+1)/(2^13-1)) carried by the key scale, sigma 1."""
    delta = float(np.log((2.0 ** 13 + 1) / (2.0 ** 13 - 1)))
    q = np.zeros(D); q[0] = 1.0
    kA = np.zeros(D, np.int8); kA[0] = 1
    kB = np.zeros(D, np.int8)
    vA = np.zeros(D, np.int8); vA[0] = 127
    vB = np.zeros(D, np.int8); vB[0] = -127
    return two_candidate(q, kA, kB, vA, vB, k_scale=delta, v_scale=32.0, sigma=1.0, spread=spread)


def large_common_logit_case(sigma: float, spread: bool = False) -> SparseCase:
    """Raw dot products 8290560 and 8290560.5 (head_dim 256: query channel 0 is
    0.5, channels 1..255 are 256; key codes 127 on channels 1..255 and 0 / 1 on
    channel 0); values 0 and 1 on channel 0."""
    D = 256
    q = np.full(D, 256.0); q[0] = 0.5
    kA = np.full(D, 127, np.int8); kA[0] = 0
    kB = np.full(D, 127, np.int8); kB[0] = 1
    vA = np.zeros(D, np.int8)
    vB = np.zeros(D, np.int8); vB[0] = 1
    return two_candidate(q, kA, kB, vA, vB, k_scale=1.0, v_scale=1.0, sigma=sigma, spread=spread)


def tiny_probability_case(q0: float, v_code: int, v_scale: float, D: int = 64,
                          spread: bool = False) -> SparseCase:
    """One query channel q0, unit key scale, key codes {0, -1}, sigma 1/16
    (scores {0, -q0/16}); value code ``v_code`` on the deep candidate only."""
    q = np.zeros(D); q[0] = q0
    kA = np.zeros(D, np.int8)
    kB = np.zeros(D, np.int8); kB[0] = -1
    vA = np.zeros(D, np.int8)
    vB = np.zeros(D, np.int8); vB[0] = v_code
    return two_candidate(q, kA, kB, vA, vB, k_scale=1.0, v_scale=v_scale, sigma=1.0 / 16.0,
                         spread=spread)


def query_folding_case(spread: bool = False) -> SparseCase:
    """Per-channel key scales 32768 and 32766 on query channels +1 and -1: the
    products Q * k_scale are 32768 and -32766, which fp16 rounds to 32768 and
    -32768.  Key codes 8 on both channels for candidate A, 0 for B; sigma 1:
    logits 16 and 0 (0 and 0 after the rounding).  Value code 1 on channel 0
    for A."""
    D = 64
    q = np.zeros(D); q[0], q[1] = 1.0, -1.0
    kA = np.zeros(D, np.int8); kA[0] = kA[1] = 8
    kB = np.zeros(D, np.int8)
    vA = np.zeros(D, np.int8); vA[0] = 1
    vB = np.zeros(D, np.int8)
    c = two_candidate(q, kA, kB, vA, vB, k_scale=1.0, v_scale=1.0, sigma=1.0, spread=spread)
    ks = np.ones((1, D), np.float32)
    ks[0, 0], ks[0, 1] = 32768.0, 32766.0
    c.k_scale = ks
    c.v_scale = np.ones((1, D), np.float32)
    c.scale_kind = SCALE_PER_CHANNEL
    c.meta = dict(name="query folding", spread=spread)
    return c
