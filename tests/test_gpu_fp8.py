"""The float8 e4m3fn cache on the GPU: the exact in-register conversion, paged
decode against the FP64 oracle, and quantize-on-write bit-exact.

[onnxruntime PR 29912, Schema: cache element type float8e4m3fn; CUDA kernels:
paged decode with on-the-fly dequantisation, ReshapeAndCache quantizes on
write; the int8 and fp8 caches are measured side by side.]
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_close_oracle, assert_lse_close, assert_lse_oracle, assert_split_close,
                     dev, oracle_paged, paged_bound, paged_to_device, run_paged)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()
    return K


def test_fp8_to_fp16_exhaustive(K):
    codes = np.tile(np.arange(256, dtype=np.uint8), 4)
    got = K.fp8_to_fp16(dev(codes)).cpu().numpy().astype(np.float64)
    want = np.array([oracle.e4m3fn_value(c) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    np.testing.assert_array_equal(got[fin], want[fin])
    np.testing.assert_array_equal(np.signbit(got[fin]), np.signbit(want[fin]))


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("kind", [W.SCALE_PER_CHANNEL, W.SCALE_PER_TENSOR])
def test_paged_decode_fp8_ragged(K, bs, kind):
    lens = [0, 1, 15, 16, 17, 300, 511, 2000]
    c = W.random_paged(seed=50 + bs + kind, B=len(lens), Hq=32, Hkv=8, D=128, bs=bs,
                       max_blocks=512 // bs, lens=lens, scale_kind=kind, sink=True, cache="fp8")
    assert c.k_cache.dtype == np.uint8
    ref_o, ref_l = oracle_paged(c)
    d = paged_to_device(c)
    o, l, slots = run_paged(c, d, slots=True)
    assert_close_oracle(o, ref_o, "auto")
    assert_lse_oracle(l, ref_l, paged_bound(c))
    np.testing.assert_array_equal(slots, oracle.paged_slots(c.block_table, c.seq_lens, bs))
    o1, l1 = run_paged(c, d, num_splits=1, chunk=512)
    for ns, ch in [(32, 16), (3, 176)]:
        o_s, l_s = run_paged(c, d, num_splits=ns, chunk=ch)
        assert_close_oracle(o_s, ref_o, f"{ns} splits")
        assert_split_close(o_s, o1, f"{ns} splits")
        assert_lse_close(l_s, l1, 1e-4)


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 8, 2), (64, 16, 1), (128, 12, 1), (256, 8, 2),
                                      (256, 16, 1)])
def test_paged_decode_fp8_head_dims(K, D, Hq, Hkv):
    c = W.random_paged(seed=D + Hq, B=3, Hq=Hq, Hkv=Hkv, D=D, bs=16, max_blocks=40,
                       lens=[640, 100, 33], sink=True, cache="fp8")
    ref_o, ref_l = oracle_paged(c)
    for ns, ch in [(0, 0), (1, 640), (10, 64)]:
        o, l = run_paged(c, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o, f"fp8 D {D} G {Hq // Hkv} splits {ns}")
        assert_lse_oracle(l, ref_l, paged_bound(c))


def test_paged_decode_fp8_softcap_and_window(K):
    c = W.random_paged(seed=77, B=5, Hq=16, Hkv=2, D=128, bs=16, max_blocks=32,
                       lens=[0, 9, 200, 512, 700], sink=True, cache="fp8")
    for softcap, window in [(1.5, -1), (0.0, 50), (2.0, 130)]:
        ref_o, ref_l = oracle_paged(c, softcap, window)
        for ns, ch in [(0, 0), (1, 512), (5, 32)]:
            if ns * ch and ns * ch < K.window_span(512, window):
                continue
            o, l = run_paged(c, num_splits=ns, chunk=ch, softcap=softcap, window=window)
            assert_close_oracle(o, ref_o, f"cap {softcap} window {window} ns {ns}")
            assert_lse_oracle(l, ref_l, paged_bound(c))


def test_deep_context_fp8_chunks_vs_single_split(K):
    c = W.deep_context(seed=4, cache="fp8", B=4, cap=1024, live=650)
    ref_o, _ = oracle_paged(c)
    o1, l1 = run_paged(c, num_splits=1, chunk=1024)
    assert_close_oracle(o1, ref_o, "single split")
    for ch in (128, 256, 512):
        o, l = run_paged(c, num_splits=-(-1024 // ch), chunk=ch)
        assert_split_close(o, o1, f"chunk {ch}")
        assert_lse_close(l, l1, 1e-4)


@pytest.mark.parametrize("kind", [W.SCALE_PER_TENSOR, W.SCALE_PER_CHANNEL])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_fp8_codes_bit_exact(K, kind, D):
    rng = np.random.default_rng(100 + D + kind)
    nb, bs, Hkv, T = 30, 16, 2, 200
    kc = rng.integers(0, 256, size=(nb, bs, Hkv, D)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(nb, bs, Hkv, D)).astype(np.uint8)
    # magnitudes across the e4m3fn range (subnormal to saturated), both signs
    kn = (np.exp2(rng.uniform(-16, 12, size=(T, Hkv, D))) *
          rng.choice([-1, 1], size=(T, Hkv, D))).astype(np.float16)
    vn = (rng.standard_normal((T, Hkv, D)) * 3).astype(np.float16)
    # exact midpoints at unit scale (ties to even), saturation, non-finite,
    # a negative value that rounds to zero
    kn[0, 0, :12] = np.array([1.0625, 1.1875, -1.0625, 0.0029296875, 460, 500, -70000.0, np.nan,
                              np.inf, -np.inf, -0.0004, 448], np.float16)
    if kind == W.SCALE_PER_TENSOR:
        ks, vs = np.array([1.0], np.float32), np.array([0.0173], np.float32)
    else:
        ks = np.exp(rng.uniform(-3, 3, size=(Hkv, D))).astype(np.float32)
        ks[0, :12] = 1.0
        vs = np.exp(rng.uniform(-5, 0, size=(Hkv, D))).astype(np.float32)
    slots = rng.permutation(nb * bs)[:T].astype(np.int32)
    slots[3] = -1
    slots[7] = nb * bs  # out of the pool
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd, vd = dev(kc), dev(vc)
    K.reshape_and_cache(dev(kn), dev(vn), dev(slots), kd, vd, dev(ks), dev(vs), kind, flags=flags)
    torch.cuda.synchronize()
    k_ref, v_ref = oracle.reshape_and_cache(kn, vn, slots, kc, vc, ks, vs, kind)
    got_k = kd.cpu().numpy()
    bad = np.argwhere(got_k != k_ref)
    assert bad.size == 0, f"{len(bad)} K codes differ, first at {bad[0]}: " \
        f"got {got_k[tuple(bad[0])]:#04x} want {k_ref[tuple(bad[0])]:#04x}"
    np.testing.assert_array_equal(vd.cpu().numpy(), v_ref)
    assert int(flags.item()) & 0x8


def test_decode_over_an_fp8_cache_written_on_the_device(K):
    c = W.random_paged(seed=23, B=4, Hq=16, Hkv=4, D=128, bs=16, max_blocks=32,
                       lens=[100, 257, 31, 500], sink=True, spare_blocks=6, cache="fp8")
    rng = np.random.default_rng(4)
    kn = rng.standard_normal((4, 4, 128)).astype(np.float16)
    vn = rng.standard_normal((4, 4, 128)).astype(np.float16)
    slots = np.array([c.block_table[b, int(L) // 16] * 16 + int(L) % 16
                      for b, L in enumerate(c.seq_lens)], np.int32)
    kd, vd = dev(c.k_cache), dev(c.v_cache)
    K.reshape_and_cache(dev(kn), dev(vn), dev(slots), kd, vd, dev(c.k_scale), dev(c.v_scale),
                        c.scale_kind)
    k_ref, v_ref = oracle.reshape_and_cache(kn, vn, slots, c.k_cache, c.v_cache, c.k_scale,
                                            c.v_scale, c.scale_kind)
    np.testing.assert_array_equal(kd.cpu().numpy(), k_ref)
    np.testing.assert_array_equal(vd.cpu().numpy(), v_ref)
    c2 = dataclasses.replace(c, k_cache=k_ref, v_cache=v_ref, seq_lens=c.seq_lens + 1)
    ref_o, ref_l = oracle_paged(c2)
    d = dict(q=dev(c2.q), k=kd, v=vd, ks=dev(c2.k_scale), vs=dev(c2.v_scale),
             bt=dev(c2.block_table), lens=dev(c2.seq_lens), sink=dev(c2.sink))
    o, l = run_paged(c2, d, num_splits=0)
    assert_close_oracle(o, ref_o, "decode after fp8 quantize-on-write")
    assert_lse_oracle(l, ref_l, paged_bound(c2))
