"""Parity of the paged decode's softcap and sliding-window options with the oracle.

[onnxruntime PR 29912, CUDA kernels: the paged decode kernel has native
head-sink, softcap, sliding-window and on-the-fly cache dequantisation.]
Outputs and lse against the FP64 oracle element by element; the windowed split
partition through the partials themselves; the debug slot table bit-exact;
capture in a CUDA graph with live lengths that change between replays.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_close_oracle, assert_lse_close, assert_lse_oracle, assert_split_close,
                     dev, lse_bound, oracle_paged, paged_to_device, run_paged)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()


def _bound(c):
    return lse_bound(c.q, c.k_scale, c.scale_kind, c.k_cache.shape[2], c.sigma,
                     fp16_cache=c.k_cache.dtype == np.float16)


LENS = [0, 1, 15, 16, 17, 300, 511, 2000]   # the last exceeds the cap 512 (clamped)


@pytest.mark.parametrize("softcap,window", [
    (0.0, 0), (0.0, 1), (0.0, 15), (0.0, 16), (0.0, 17), (0.0, 100), (0.0, 5000),
    (1.0, -1), (2.0, -1), (30.0, -1), (5.0, 300), (1.5, 16)])
@pytest.mark.parametrize("kind", [W.SCALE_PER_CHANNEL, W.SCALE_PER_TENSOR])
def test_paged_softcap_and_window(softcap, window, kind):
    import int8_kv_cache_gb300 as K
    c = W.random_paged(seed=31 + kind, B=len(LENS), Hq=32, Hkv=8, D=128, bs=16, max_blocks=32,
                       lens=LENS, scale_kind=kind, sink=True)
    # sigma = 1/sqrt(D) gives scores of about one unit, which caps of 1 and 2
    # bend strongly; a larger sigma would only scale up the fp16 rounding of
    # the folded query beyond what the output tolerance is stated for
    ref_o, ref_l = oracle_paged(c, softcap, window)
    d = paged_to_device(c)
    span = K.window_span(512, window)
    o, l, slots = run_paged(c, d, slots=True, softcap=softcap, window=window)
    assert_close_oracle(o, ref_o, "auto")
    assert_lse_oracle(l, ref_l, _bound(c))
    np.testing.assert_array_equal(slots, oracle.paged_slots(c.block_table, c.seq_lens, 16, window))
    one = -(-span // 16) * 16
    o1, l1 = run_paged(c, d, num_splits=1, chunk=one, softcap=softcap, window=window)
    assert_close_oracle(o1, ref_o, "1 split")
    for ch in (16, 48, 128):
        ns = -(-span // ch)
        if ns > 32:
            continue
        o_s, l_s, sl = run_paged(c, d, num_splits=ns, chunk=ch, slots=True, softcap=softcap,
                                 window=window)
        assert_close_oracle(o_s, ref_o, f"{ns} x {ch}")
        assert_split_close(o_s, o1, f"{ns} x {ch}")
        assert_lse_close(l_s, l1, 1e-4)
        np.testing.assert_array_equal(sl, slots)


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 16, 2), (256, 12, 1), (128, 16, 1)])
@pytest.mark.parametrize("cache", ["int8", "fp16"])
def test_paged_variants_head_dims_and_fp16_cache(D, Hq, Hkv, cache):
    c = W.random_paged(seed=D + Hq, B=4, Hq=Hq, Hkv=Hkv, D=D, bs=32, max_blocks=24,
                       lens=[700, 64, 33, 0], cache=cache, sink=True)
    for softcap, window in [(1.0, -1), (0.0, 77), (2.0, 250)]:
        ref_o, ref_l = oracle_paged(c, softcap, window)
        for ns, ch in [(0, 0), (1, 768), (6, 128)]:
            o, l = run_paged(c, num_splits=ns, chunk=ch, softcap=softcap, window=window)
            assert_close_oracle(o, ref_o, f"{cache} D {D} cap {softcap} w {window} ns {ns}")
            assert_lse_oracle(l, ref_l, _bound(c))


@pytest.mark.parametrize("softcap,window,ns,chunk", [(0.0, 40, 4, 16), (1.0, 100, 3, 48),
                                                     (0.0, -1, 8, 64), (1.5, 5000, 4, 128)])
def test_windowed_partials_follow_the_window_partition(softcap, window, ns, chunk):
    c = W.random_paged(seed=5, B=5, Hq=16, Hkv=4, D=128, bs=16, max_blocks=32,
                       lens=[0, 20, 130, 301, 512], sink=False)
    m, l, acc = run_paged(c, num_splits=ns, chunk=chunk, softcap=softcap, window=window,
                          partials=True)
    rm, rl, ra = oracle.paged_split_partials(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                             c.scale_kind, c.block_table, c.seq_lens, c.sigma,
                                             ns, chunk, softcap=softcap, window=window)
    B, Hq, Hkv, G, D = 5, 16, 4, 4, 128
    rm = rm.reshape(B, Hkv, G, ns).transpose(0, 1, 3, 2).reshape(B * Hkv, ns, G)
    rl = rl.reshape(B, Hkv, G, ns).transpose(0, 1, 3, 2).reshape(B * Hkv, ns, G)
    ra = ra.reshape(B, Hkv, G, ns, D).transpose(0, 1, 3, 2, 4).reshape(B * Hkv, ns, G, D)
    bnd = _bound(c).reshape(B, Hkv, G)[:, :, None, :].repeat(ns, axis=2).reshape(B * Hkv, ns, G)
    empty = np.isneginf(rm)
    assert np.array_equal(np.isneginf(m), empty), "empty-split pattern differs"
    assert np.all(l[empty] == 0)
    live = ~empty
    assert np.all(np.abs(m[live] - rm[live]) <= bnd[live] + 1e-6 * np.abs(rm[live]))
    # the sums and accumulators are taken relative to each side's own maximum
    # (a per-score error e moves ln l by at most e: the lse bound applies)
    lr = l[live] * np.exp(m[live] - rm[live])
    assert np.all(np.abs(np.log(lr / rl[live])) <= bnd[live] + 1e-5)
    assert_close_oracle(acc[live] / l[live][:, None], ra[live] / rl[live][:, None],
                        "normalised partial")


def test_windowed_decode_in_a_cuda_graph_with_changing_lengths():
    import int8_kv_cache_gb300 as K
    lens_a = [300, 17, 512, 1]
    lens_b = [511, 0, 40, 260]
    # the table covers both sets of lengths
    c = W.random_paged(seed=12, B=4, Hq=16, Hkv=2, D=128, bs=16, max_blocks=32,
                       lens=np.maximum(lens_a, lens_b), sink=True)
    d = paged_to_device(c)
    softcap, window = 2.0, 100
    span = K.window_span(512, window)
    ns, ch, wsb, _ = K.decode_plan(K.PATH_PAGED, K.CACHE_INT8, span, 4, 16, 2, 128, K.GEOM_WAVE)
    assert ns * ch >= span and ns * ch < 512
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    out = torch.empty((4, 16, 128), dtype=torch.float16, device="cuda")
    lse = torch.empty((4, 16), dtype=torch.float32, device="cuda")

    def call():
        K.paged_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["bt"], d["lens"],
                       c.sigma, d["sink"], num_splits=ns, chunk=ch, workspace=ws, out=out,
                       lse=lse, softcap=softcap, window=window)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # first call outside capture (per-device attribute setup)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for lens in (lens_a, lens_b):
        c.seq_lens = np.asarray(lens, dtype=np.int32)
        d["lens"].copy_(dev(c.seq_lens))
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle_paged(c, softcap, window)
        assert_close_oracle(out.float().cpu().numpy().astype(np.float64), ref_o, f"lens {lens}")
        assert_lse_oracle(lse.cpu().numpy().astype(np.float64), ref_l, _bound(c))
