"""Balanced pieces of the paged decode (num_splits partial slots, chunk 0):
the grid and the workspace come from the arguments, the pieces of each row's
live range are cut on the device from all live lengths.  Against the FP64
oracle on ragged batches (every cache kind, sink, softcap, sliding window,
empty and over-long rows, one row), against the same call with the wave
rule's fixed chunks, across CUDA-graph replays with new lengths, with a
NaN-filled workspace (the unused slots must be marked empty), and the
argument rules."""
import numpy as np
import pytest
import torch

import int8_kv_cache_gb300 as K
import workloads as W
from helpers import (assert_close_oracle, assert_lse_close, assert_lse_oracle, assert_split_close,
                     oracle_paged, paged_bound, paged_to_device, run_paged)

pytestmark = pytest.mark.gpu


def _slots(c, window=-1):
    B, Hq, D = c.q.shape
    nb, bs, Hkv, _ = c.k_cache.shape
    dt = {np.dtype(np.float16): K.CACHE_FP16, np.dtype(np.uint8): K.CACHE_FP8}.get(
        c.k_cache.dtype, K.CACHE_INT8)
    cap = c.block_table.shape[1] * bs
    ns, chunk, wsb, _ = K.decode_plan(K.PATH_PAGED, dt, K.window_span(cap, window), B, Hq, Hkv, D,
                                      K.GEOM_BALANCED)
    assert chunk == 0 and 2 <= ns <= 32
    assert wsb == K.split_workspace_bytes(B * Hkv, ns, Hq // Hkv, D)
    return ns


@pytest.mark.parametrize("cache", ["int8", "fp8", "fp16"])
@pytest.mark.parametrize("seed,B,lens_hi", [(0, 16, 3000), (1, 5, 4096), (2, 40, 1500)])
def test_ragged_batch_matches_the_oracle(cache, seed, B, lens_hi):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, lens_hi + 1, size=B)
    c = W.random_paged(seed=seed, B=B, Hq=32, Hkv=8, D=128, bs=16, max_blocks=256, lens=lens,
                       sink=True, cache=cache)
    ns = _slots(c)
    ref_o, ref_l = oracle_paged(c)
    o, l = run_paged(c, num_splits=ns, chunk=0)
    assert_close_oracle(o, ref_o, f"balanced {cache}")
    assert_lse_oracle(l, ref_l, paged_bound(c))
    # the same call with the wave rule's chunks: split against split
    ow, lw = run_paged(c)
    assert_split_close(o, ow, "balanced vs wave rule")
    assert_lse_close(l, lw, 1e-4)


@pytest.mark.parametrize("softcap,window", [(30.0, -1), (0.0, 300), (30.0, 1023)])
def test_softcap_and_window(softcap, window):
    lens = [5, 700, 4096, 1500, 2999, 64, 3333, 17]
    c = W.random_paged(seed=7, B=len(lens), Hq=16, Hkv=2, D=128, bs=16, max_blocks=256, lens=lens,
                       sink=True)
    ns = _slots(c, window)
    ref_o, ref_l = oracle_paged(c, softcap=softcap, window=window)
    o, l = run_paged(c, num_splits=ns, chunk=0, softcap=softcap, window=window)
    assert_close_oracle(o, ref_o, "balanced softcap/window")
    assert_lse_oracle(l, ref_l, paged_bound(c))


def test_empty_clamped_and_single_rows():
    # a row of length 0 (O = 0, lse = -inf), one past the capacity (clamped,
    # flagged), and a batch of one row
    lens = [0, 5000, 1, 4096, 300]
    c = W.random_paged(seed=9, B=5, Hq=8, Hkv=2, D=256, bs=16, max_blocks=256, lens=lens)
    ns = _slots(c)
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_o, ref_l = oracle_paged(c)
    o, l = run_paged(c, num_splits=ns, chunk=0, flags=f)
    assert int(f.item()) & K.FLAG_LEN_CLAMPED
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    assert_close_oracle(o, ref_o, "balanced edge rows")
    assert_lse_oracle(l, ref_l, paged_bound(c))
    c1 = W.random_paged(seed=10, B=1, Hq=16, Hkv=2, D=128, bs=16, max_blocks=512, lens=[8000])
    ns1 = _slots(c1)
    ref_o, ref_l = oracle_paged(c1)
    o, l = run_paged(c1, num_splits=ns1, chunk=0)
    assert_close_oracle(o, ref_o, "balanced one row")
    assert_lse_oracle(l, ref_l, paged_bound(c1))


def test_graph_replays_follow_new_lengths():
    # the launch depends on the arguments only: a graph captured once serves
    # other live lengths when the lengths buffer changes between replays
    B = 12
    rng = np.random.default_rng(3)
    lens_a = rng.integers(1, 4096, size=B)
    lens_b = rng.integers(1, 4096, size=B)
    lens_b[0] = 4096
    # blocks for the longer of the two lengths of every row
    ca = W.random_paged(seed=11, B=B, Hq=32, Hkv=8, D=128, bs=16, max_blocks=256,
                        lens=np.maximum(lens_a, lens_b), sink=True)
    d = paged_to_device(ca)
    ns = _slots(ca)
    Hq, D = ca.q.shape[1], ca.q.shape[2]
    wsb = K.split_workspace_bytes(B * 8, ns, Hq // 8, D)
    ws = torch.full((wsb // 4,), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.empty_like(d["q"])
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        K.paged_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], ca.scale_kind, d["bt"],
                       d["lens"], ca.sigma, d["sink"], num_splits=ns, chunk=0, workspace=ws,
                       out=out, lse=lse)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for lens in (lens_b, lens_a):
        d["lens"].copy_(torch.from_numpy(lens.astype(np.int32)))
        g.replay()
        torch.cuda.synchronize()
        ca.seq_lens = lens.astype(np.int32)
        ref_o, ref_l = oracle_paged(ca)
        o = out.float().cpu().numpy().astype(np.float64)
        l = lse.cpu().numpy().astype(np.float64)
        assert_close_oracle(o, ref_o, "balanced graph replay")
        assert_lse_oracle(l, ref_l, paged_bound(ca))


def test_argument_rules():
    c = W.random_paged(seed=12, B=4, Hq=8, Hkv=2, D=128, bs=16, max_blocks=64, lens=[10, 20, 30, 40])
    d = paged_to_device(c)
    ws = torch.zeros(1 << 20, dtype=torch.float32, device="cuda")
    so = torch.zeros((4, 64 * 16), dtype=torch.int32, device="cuda")
    with pytest.raises(K.Int8KVError):  # the debug slots need the fixed chunks
        K.paged_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["bt"], d["lens"],
                       c.sigma, num_splits=4, chunk=0, workspace=ws, slots_out=so)
    with pytest.raises(K.Int8KVError):  # more slots than MAX_SPLITS
        K.paged_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["bt"], d["lens"],
                       c.sigma, num_splits=33, chunk=0, workspace=ws)
    with pytest.raises(K.Int8KVError):  # the sparse path has no balanced mode
        K.decode_plan(K.PATH_DSA, K.CACHE_INT8, 2048, 8, 24, 2, 256, K.GEOM_BALANCED)
    cb = W.random_paged(seed=13, B=129, Hq=8, Hkv=2, D=128, bs=16, max_blocks=4,
                        lens=np.full(129, 40))
    db = paged_to_device(cb)
    with pytest.raises(K.Int8KVError):  # more than 128 rows
        K.paged_decode(db["q"], db["k"], db["v"], db["ks"], db["vs"], cb.scale_kind, db["bt"],
                       db["lens"], cb.sigma, num_splits=4, chunk=0, workspace=ws)
