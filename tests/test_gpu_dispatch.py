"""Longest-first dispatch of the paged decode, against the FP64 oracle.

Paged calls whose chunks hold at least 2048 tokens (batches of up to 128 rows)
hand the (unit, split) items to the CTAs longest chunk first instead of in
split-major order.  Only which CTA computes which split changes, so every
output, lse and split partial must still be the oracle's.  The lengths put
items in every class the order distinguishes: full chunks, partial chunks in
each quarter of a chunk, empty chunks, an empty row and a length beyond the
capacity (clamped).  [onnxruntime PR 29912, CUDA kernels: split-K paged
decode; onnx-genai PR 1350: the split count comes from the capacity and the
row count only, so a captured graph replays with other lengths.]
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_close_oracle, assert_lse_oracle, lse_bound, oracle_paged,
                     paged_to_device, run_paged)

pytestmark = pytest.mark.gpu

CHUNK = 2048
# cap 8192 = 4 chunks: rows with 0..4 full chunks and partial chunks of
# 1, 44, 1104, 2044, 2047 tokens (quarters 0, 0, 2, 3, 3), one empty row and
# one row beyond the cap
LENS = [0, 1, 2047, 2048, 2049, 4095, 4096, 4140, 5200, 6140, 8192, 9000]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()


def _bound(c):
    return lse_bound(c.q, c.k_scale, c.scale_kind, c.k_cache.shape[2], c.sigma,
                     fp16_cache=c.k_cache.dtype == np.float16,
                     code_max=448.0 if c.k_cache.dtype == np.uint8 else 128.0)


def _case(lens, cache="int8", seed=31, Hq=16, Hkv=2):
    return W.random_paged(seed=seed, B=len(lens), Hq=Hq, Hkv=Hkv, D=128, bs=16, max_blocks=512,
                          lens=lens, sink=True, cache=cache)


def _check_outputs(c, o, lse, window=-1):
    ref_o, ref_lse = oracle_paged(c, window=window)
    assert_close_oracle(o, ref_o, "output")
    assert_lse_oracle(lse, ref_lse, _bound(c), "lse")


def _check_partials(c, ns, window=-1):
    B, Hq, D = c.q.shape
    Hkv = c.k_cache.shape[2]
    G = Hq // Hkv
    m, l, acc = run_paged(c, num_splits=ns, chunk=CHUNK, window=window, partials=True)
    rm, rl, ra = oracle.paged_split_partials(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                             c.scale_kind, c.block_table, c.seq_lens, c.sigma,
                                             ns, CHUNK, window=window)
    rm = rm.reshape(B, Hkv, G, ns).transpose(0, 1, 3, 2).reshape(B * Hkv, ns, G)
    rl = rl.reshape(B, Hkv, G, ns).transpose(0, 1, 3, 2).reshape(B * Hkv, ns, G)
    ra = ra.reshape(B, Hkv, G, ns, D).transpose(0, 1, 3, 2, 4).reshape(B * Hkv, ns, G, D)
    bnd = _bound(c).reshape(B, Hkv, G)[:, :, None, :].repeat(ns, axis=2).reshape(B * Hkv, ns, G)
    empty = np.isneginf(rm)
    assert np.array_equal(np.isneginf(m), empty), "empty-split pattern differs"
    assert np.all(l[empty] == 0)
    live = ~empty
    assert np.all(np.abs(m[live] - rm[live]) <= bnd[live] + 1e-6 * np.abs(rm[live]))
    lr = l[live] * np.exp(m[live] - rm[live])
    assert np.all(np.abs(np.log(lr / rl[live])) <= bnd[live] + 1e-5)
    assert_close_oracle(acc[live] / l[live][:, None], ra[live] / rl[live][:, None],
                        "normalised partial")


@pytest.mark.parametrize("cache", ["int8", "fp8", "fp16"])
def test_ragged_rows_every_item_class(cache):
    c = _case(LENS, cache=cache)
    o, lse = run_paged(c, num_splits=4, chunk=CHUNK)
    _check_outputs(c, o, lse)
    _check_partials(c, 4)


def test_window_with_long_chunks():
    # window 3500: span min(8192, 3516) = 3516 -> 2 chunks of 2048 counted from
    # the window start
    c = _case(LENS, seed=32)
    o, lse = run_paged(c, num_splits=2, chunk=CHUNK, window=3500)
    _check_outputs(c, o, lse, window=3500)
    _check_partials(c, 2, window=3500)


@pytest.mark.parametrize("B", [32, 33, 100, 128, 129])
def test_batches_up_to_128_rows_and_one_more(B):
    # up to 128 rows (one to four rows per lane): the dispatch ranks the
    # batch; 129 rows: split-major order
    lens = W.make_rng(33).integers(0, 9200, size=B)
    c = _case(lens, seed=34, Hq=8, Hkv=1)
    o, lse = run_paged(c, num_splits=4, chunk=CHUNK)
    _check_outputs(c, o, lse)


def test_single_split_rows_ordered_by_length():
    # one split of the whole capacity: the items are the units, longest first
    c = _case([10, 8000, 0, 5000, 1400, 8192], seed=35)
    o, lse = run_paged(c, num_splits=1, chunk=8192)
    _check_outputs(c, o, lse)


def test_captured_graph_replays_with_other_lengths():
    """The order is decided on the device from the live lengths: one captured
    launch serves two different batches."""
    import int8_kv_cache_gb300 as K
    lens_a = [4096, 10, 6000, 0, 8192, 3000]
    lens_b = [1, 8192, 2048, 5200, 60, 6666]
    c = _case(np.maximum(lens_a, lens_b), seed=36)
    d = paged_to_device(c)
    B, Hq, D = c.q.shape
    Hkv = c.k_cache.shape[2]
    ns = 4
    wsb = K.split_workspace_bytes(B * Hkv, ns, Hq // Hkv, D)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.float16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    lens_dev = d["lens"]
    s = torch.cuda.Stream()

    def call():
        K.paged_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["bt"], lens_dev,
                       c.sigma, d["sink"], num_splits=ns, chunk=CHUNK, workspace=ws, out=out,
                       lse=lse, stream=s)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for lens in (lens_a, lens_b):
        lens_dev.copy_(torch.tensor(lens, dtype=torch.int32))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        ci = W.PagedCase(q=c.q, k_cache=c.k_cache, v_cache=c.v_cache, k_scale=c.k_scale,
                         v_scale=c.v_scale, scale_kind=c.scale_kind, block_table=c.block_table,
                         seq_lens=np.asarray(lens, np.int32), sigma=c.sigma, sink=c.sink)
        _check_outputs(ci, out.float().cpu().numpy().astype(np.float64),
                       lse.cpu().numpy().astype(np.float64))
