"""Parity of the CUDA path (through the C ABI) with the FP64 oracle.

Small and medium cases, element by element: the tiny decode, sparse-candidate
decode sweeps (group sizes 4/6/12/16, list lengths around the 64-candidate
tile, invalid entries, split counts), paged decode (ragged lengths, empty and
over-long sequences, permuted block tables, fp16 cache), prefill, the analytic
two-candidate cases, the combine on its own, the exact conversion and the
device flags.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_close_oracle, assert_lse_close, assert_lse_oracle, assert_split_close,
                     dev, lse_bound, oracle_dsa, oracle_paged, paged_to_device, run_dsa,
                     run_paged, sparse_to_device)


def bound_of(c):
    """lse tolerance against the oracle for a sparse or paged case."""
    if hasattr(c, "k_codes"):
        return lse_bound(c.q, c.k_scale, c.scale_kind, c.k_codes.shape[1], c.sigma)
    return lse_bound(c.q, c.k_scale, c.scale_kind, c.k_cache.shape[2], c.sigma,
                     fp16_cache=c.k_cache.dtype == np.float16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()


def test_int8_to_fp16_exhaustive():
    import int8_kv_cache_gb300 as K
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    x = np.tile(codes, 64)  # 16384 bytes, every code in every byte position
    got = K.int8_to_fp16(dev(x)).cpu().numpy()
    np.testing.assert_array_equal(got.astype(np.float32), x.astype(np.float32))
    assert got.dtype == np.float16


# --------------------------------------------------------------------------
# tiny decode (1 sequence, 4/1 heads, head_dim 64, 128 tokens), splits 1 and 4
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kind", [W.SCALE_PER_CHANNEL, W.SCALE_PER_TENSOR])
def test_tiny_decode_paged_splits_1_and_4(kind):
    c = W.tiny_decode(seed=0, scale_kind=kind)
    ref_o, ref_l = oracle_paged(c)
    o1, l1 = run_paged(c, num_splits=1, chunk=128)
    o4, l4 = run_paged(c, num_splits=4, chunk=32)
    assert_close_oracle(o1, ref_o, "1 split")
    assert_close_oracle(o4, ref_o, "4 splits")
    assert_lse_oracle(l1, ref_l, bound_of(c))
    assert_lse_oracle(l4, ref_l, bound_of(c))
    assert_split_close(o4, o1, "tiny")
    assert_lse_close(l4, l1, 1e-4)


def test_tiny_decode_as_sparse_list():
    c = W.tiny_decode(seed=0)
    kc = c.k_cache.reshape(128, 1, 64)
    vc = c.v_cache.reshape(128, 1, 64)
    s = W.SparseCase(q=c.q, k_codes=kc, v_codes=vc, k_scale=c.k_scale, v_scale=c.v_scale,
                     scale_kind=c.scale_kind, idx=np.arange(128, dtype=np.int32).reshape(1, 128),
                     sigma=c.sigma)
    ref_o, ref_l = oracle_dsa(s)
    for ns, ch in [(1, 128), (4, 32), (2, 64)]:
        o, l = run_dsa(s, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o, f"splits {ns}")
        assert_lse_oracle(l, ref_l, bound_of(s))


# --------------------------------------------------------------------------
# sparse-candidate decode sweep (the page's: rows x heads x selected x splits)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 3, 8])
@pytest.mark.parametrize("Hq", [8, 12, 24, 32])
@pytest.mark.parametrize("max_sel", [1, 65, 509])
def test_dsa_decode_sweep(S, Hq, max_sel):
    c = W.random_sparse(seed=S * 1000 + Hq * 10 + max_sel, S=S, Hq=Hq, Hkv=2, D=256, N=700,
                        max_sel=max_sel, invalid_frac=0.2, sink=(Hq == 24), sigma=1.0 / 16)
    ref_o, ref_l = oracle_dsa(c)
    d = sparse_to_device(c)
    o_auto, l_auto = run_dsa(c, d, num_splits=0)
    assert_close_oracle(o_auto, ref_o, "auto splits")
    assert_lse_oracle(l_auto, ref_l, bound_of(c))
    o1, l1 = run_dsa(c, d, num_splits=1, chunk=((max_sel + 15) // 16) * 16)
    assert_close_oracle(o1, ref_o, "1 split")
    # 1 and 3 tiles (64 candidates) per split; a split may be empty
    for tps in (1, 3):
        ch = 64 * tps
        ns = max(1, -(-max_sel // ch))
        o, l = run_dsa(c, d, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o, f"{tps} tiles per split")
        assert_split_close(o, o1, f"{tps} tiles per split")
        assert_lse_close(l, l1, 1e-4)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 5, 8, 16])
def test_dsa_decode_head_dims(D, G):
    c = W.random_sparse(seed=D + G, S=2, Hq=2 * G, Hkv=2, D=D, N=333, max_sel=200,
                        invalid_frac=0.1, scale_kind=W.SCALE_PER_TENSOR, sink=True)
    ref_o, ref_l = oracle_dsa(c)
    for ns, ch in [(0, 0), (1, 208), (7, 32)]:
        o, l = run_dsa(c, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o, f"D {D} G {G} splits {ns}")
        assert_lse_oracle(l, ref_l, bound_of(c))


def test_dsa_tiles_per_split_caps():
    # lists of 2048 / 2112 / 8192 candidates: every candidate reaches the merge
    for n_sel, tps in [(2048, 1), (2112, 2), (2112, 3), (8192, 1), (2048, 64)]:
        c = W.random_sparse(seed=n_sel + tps, S=1, Hq=24, Hkv=2, D=256, N=9000, max_sel=n_sel,
                            sigma=1.0 / 16)
        import int8_kv_cache_gb300 as K
        ns, ch = K.split_geometry(n_sel, 2, 304, 64, 128, 32, K.GEOM_POW2_TILES, tps)
        ref_o, ref_l = oracle_dsa(c)
        o, l = run_dsa(c, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o, f"{n_sel} candidates, {tps} tiles per split")
        assert_lse_oracle(l, ref_l, bound_of(c))


def test_dsa_empty_lists_and_all_invalid_rows():
    c = W.random_sparse(seed=5, S=3, Hq=8, Hkv=2, D=128, N=50, max_sel=40, sink=True)
    c.idx[0, :] = -1
    c.idx[1, :] = 50  # all out of range
    ref_o, ref_l = oracle_dsa(c)
    for ns, ch in [(1, 48), (3, 16)]:
        o, l = run_dsa(c, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o)
        assert np.all(o[:2] == 0) and np.all(np.isneginf(l[:2]))
        assert_lse_oracle(l, ref_l, bound_of(c))


def test_dsa_duplicates_count_twice():
    c = W.random_sparse(seed=6, S=2, Hq=4, Hkv=1, D=64, N=40, max_sel=30)
    c.idx[0, 10:20] = c.idx[0, 0]
    ref_o, ref_l = oracle_dsa(c)
    o, l = run_dsa(c, num_splits=2, chunk=16)
    assert_close_oracle(o, ref_o)
    assert_lse_oracle(l, ref_l, bound_of(c))


# --------------------------------------------------------------------------
# paged decode
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("kind", [W.SCALE_PER_CHANNEL, W.SCALE_PER_TENSOR])
def test_paged_decode_ragged(bs, kind):
    lens = [0, 1, 15, 16, 17, 300, 511, 2000]  # the last one exceeds the cap (clamped)
    c = W.random_paged(seed=bs + kind, B=len(lens), Hq=32, Hkv=8, D=128, bs=bs,
                       max_blocks=512 // bs, lens=lens, scale_kind=kind, sink=True)
    ref_o, ref_l = oracle_paged(c)
    d = paged_to_device(c)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, l, slots = run_paged(c, d, num_splits=0, slots=True, flags=flags)
    assert_close_oracle(o, ref_o, "auto")
    assert_lse_oracle(l, ref_l, bound_of(c))
    np.testing.assert_array_equal(slots, oracle.paged_slots(c.block_table, c.seq_lens, bs))
    assert int(flags.item()) & 0x1, "the over-long length must be flagged"
    o1, l1 = run_paged(c, d, num_splits=1, chunk=512)
    for ns, ch in [(32, 16), (3, 176), (5, 112)]:
        o_s, l_s, sl = run_paged(c, d, num_splits=ns, chunk=ch, slots=True)
        assert_close_oracle(o_s, ref_o, f"{ns} splits")
        assert_split_close(o_s, o1, f"{ns} splits")
        assert_lse_close(l_s, l1, 1e-4)
        np.testing.assert_array_equal(sl, slots)


@pytest.mark.parametrize("D", [64, 256])
def test_paged_decode_head_dims(D):
    c = W.random_paged(seed=D, B=3, Hq=12, Hkv=1, D=D, bs=16, max_blocks=40, lens=[640, 100, 33],
                       sink=False)
    ref_o, ref_l = oracle_paged(c)
    for ns, ch in [(0, 0), (1, 640), (10, 64)]:
        o, l = run_paged(c, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o, f"D {D} splits {ns}")
        assert_lse_oracle(l, ref_l, bound_of(c))


@pytest.mark.parametrize("D", [64, 128, 256])
def test_paged_decode_fp16_cache(D):
    c = W.random_paged(seed=7 + D, B=4, Hq=16, Hkv=2, D=D, bs=16, max_blocks=64,
                       lens=[1024, 700, 5, 0], cache="fp16", sink=True)
    ref_o, ref_l = oracle_paged(c)
    for ns, ch in [(0, 0), (1, 1024), (8, 128)]:
        o, l = run_paged(c, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o, f"fp16 cache D {D} splits {ns}")
        assert_lse_oracle(l, ref_l, bound_of(c))


def test_deep_context_small_fixed_chunks_vs_single_split():
    for cache in ("int8", "fp16"):
        c = W.deep_context(seed=3, cache=cache, B=4, cap=1024, live=650)
        ref_o, ref_l = oracle_paged(c)
        o1, l1 = run_paged(c, num_splits=1, chunk=1024)
        assert_close_oracle(o1, ref_o, cache)
        for ch in (128, 256, 512):
            o, l = run_paged(c, num_splits=-(-1024 // ch), chunk=ch)
            assert_split_close(o, o1, f"{cache} chunk {ch}")
            assert_lse_close(l, l1, 1e-4)
        o, l = run_paged(c, num_splits=0)
        assert_split_close(o, o1, f"{cache} adaptive")


def test_paged_bad_block_is_flagged_and_skipped():
    c = W.random_paged(seed=9, B=2, Hq=4, Hkv=1, D=64, bs=16, max_blocks=4, lens=[64, 64])
    good_table = c.block_table.copy()
    c.block_table[1, 2] = c.k_cache.shape[0] + 5  # out of the pool
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, l = run_paged(c, num_splits=1, chunk=64, flags=flags)
    assert int(flags.item()) & 0x4
    # sequence 0 is unaffected; sequence 1 attends its tokens outside block 2
    kf, vf = c.k_cache.reshape(-1, 1, 64), c.v_cache.reshape(-1, 1, 64)
    for b, skip in ((0, range(0)), (1, range(32, 48))):
        idx = np.array([[good_table[b, t // 16] * 16 + t % 16 for t in range(64) if t not in skip]],
                       np.int32)
        ref, _ = oracle.sparse_attention(c.q[b:b + 1], kf, vf, c.k_scale, c.v_scale, c.scale_kind,
                                         idx, c.sigma)
        assert_close_oracle(o[b:b + 1], ref, f"sequence {b}")


def _with_lens(c, lens):
    import dataclasses
    return dataclasses.replace(c, seq_lens=np.array(lens, np.int32))


# --------------------------------------------------------------------------
# prefill
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Hq,D", [(24, 256), (8, 128), (4, 64)])
def test_prefill_causal_lists(Hq, D):
    c = W.sparse_prefill(seed=1, rows=48, N=300, Hq=Hq, Hkv=2 if Hq > 4 else 1, D=D, n_sel=100)
    ref_o, ref_l = oracle_dsa(c)
    o, l = run_dsa(c, prefill=True)
    assert_close_oracle(o, ref_o, "prefill")
    assert_lse_oracle(l, ref_l, bound_of(c))


def test_prefill_literal_rows_attend_their_prefix():
    c = W.sparse_prefill(seed=2, rows=70, N=70, literal=True, n_sel=64)
    ref_o, ref_l = oracle_dsa(c)
    o, l = run_dsa(c, prefill=True)
    assert_close_oracle(o, ref_o, "literal prefill")


# --------------------------------------------------------------------------
# the analytic two-candidate cases
# --------------------------------------------------------------------------

def _both_layouts(make):
    return [make(False), make(True)]


@pytest.mark.parametrize("spread", [False, True])
def test_signed_cancellation_decode(spread):
    c = W.signed_cancellation_case(spread=spread)
    for ns, ch in [(1, 192), (3, 64)]:
        o, l = run_dsa(c, num_splits=ns, chunk=ch)
        assert abs(o[0, 0, 0] - 127.0 / 256.0) <= 2.5e-4, o[0, 0, 0]


@pytest.mark.parametrize("sigma,want", [(1.0, 1 / (1 + math.exp(-0.5))),
                                        (1.0 / 16, 1 / (1 + math.exp(-1 / 32)))])
@pytest.mark.parametrize("spread", [False, True])
def test_large_common_logit(sigma, want, spread):
    c = W.large_common_logit_case(sigma, spread=spread)
    for ns, ch in [(1, 192), (3, 64)]:
        o, l = run_dsa(c, num_splits=ns, chunk=ch)
        assert abs(o[0, 0, 0] - want) <= 2e-3 + 1e-2 * want, (ns, o[0, 0, 0], want)
        o, l = run_dsa(c, prefill=True)
        assert abs(o[0, 0, 0] - want) <= 2e-3 + 1e-2 * want


@pytest.mark.parametrize("q0,code,vs,gap", [(288.0, 100, 2.0 ** 16, 18.0),
                                            (320.0, 1, 2.0 ** 28, 20.0)])
@pytest.mark.parametrize("spread", [False, True])
def test_tiny_probability_large_value_scale(q0, code, vs, gap, spread):
    c = W.tiny_probability_case(q0, code, vs, spread=spread)
    want = code * vs * math.exp(-gap) / (1 + math.exp(-gap))
    for ns, ch in [(1, 192), (3, 64)]:
        o, l = run_dsa(c, num_splits=ns, chunk=ch)
        assert abs(o[0, 0, 0] - want) <= 2e-3 + 1e-2 * want, (ns, o[0, 0, 0], want)


# --------------------------------------------------------------------------
# the combine on its own, the flags
# --------------------------------------------------------------------------

def test_split_combine_matches_oracle():
    import int8_kv_cache_gb300 as K
    c = W.random_sparse(seed=44, S=3, Hq=12, Hkv=2, D=128, N=400, max_sel=300, invalid_frac=0.1,
                        sink=True)
    ns, ch = 5, 64
    m, l, a = oracle.sparse_split_partials(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                           c.scale_kind, c.idx, c.sigma, ns, ch)
    # oracle partials [S, Hq, ns(, D)] -> workspace layout [S*Hkv, ns, G(, D)]
    S, Hq, G = 3, 12, 6
    acc = a.reshape(S, 2, G, ns, 128).transpose(0, 1, 3, 2, 4).reshape(S * 2, ns, G, 128)
    mm = m.reshape(S, 2, G, ns).transpose(0, 1, 3, 2).reshape(S * 2, ns, G)
    ll = l.reshape(S, 2, G, ns).transpose(0, 1, 3, 2).reshape(S * 2, ns, G)
    lse = torch.empty(S * Hq, dtype=torch.float32, device="cuda")
    out = K.split_combine(dev(acc, torch.float32), dev(mm, torch.float32), dev(ll, torch.float32),
                          Hq, 2, head_sink=dev(c.sink), lse=lse)
    ref_o, ref_l = oracle.combine_all(m, l, a, c.sink)
    got = out.float().cpu().numpy().reshape(S, Hq, 128)
    assert_close_oracle(got.astype(np.float64), ref_o)
    assert_lse_close(lse.cpu().numpy().reshape(S, Hq).astype(np.float64), ref_l, 1e-5)


def test_query_range_flag():
    c = W.random_sparse(seed=3, S=1, Hq=4, Hkv=1, D=64, N=50, max_sel=20)
    c.k_scale[:] = 1e6  # Q * k_scale beyond the fp16 range
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_dsa(c, num_splits=1, chunk=32, flags=flags)
    assert int(flags.item()) & 0x2


def test_capture_in_a_cuda_graph_matches_eager():
    import int8_kv_cache_gb300 as K
    c = W.random_paged(seed=1, B=6, Hq=32, Hkv=8, D=128, bs=16, max_blocks=64,
                       lens=[1000, 17, 512, 0, 1024, 333], sink=True)
    d = paged_to_device(c)
    ns, ch, wsb, _ = K.decode_plan(K.PATH_PAGED, K.CACHE_INT8, 1024, 6, 32, 8, 128, K.GEOM_WAVE)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    out = torch.empty(6, 32, 128, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        K.paged_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["bt"], d["lens"],
                       c.sigma, d["sink"], num_splits=ns, chunk=ch, workspace=ws, out=out)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        K.paged_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["bt"], d["lens"],
                       c.sigma, d["sink"], num_splits=ns, chunk=ch, workspace=ws, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    # live lengths are read on the device: change them and replay
    d["lens"].copy_(torch.tensor([5, 1024, 0, 700, 1, 64], dtype=torch.int32))
    g.replay()
    torch.cuda.synchronize()
    ref_o, _ = oracle_paged(_with_lens(c, [5, 1024, 0, 700, 1, 64]))
    assert_close_oracle(out.float().cpu().numpy().astype(np.float64), ref_o, "replay")
