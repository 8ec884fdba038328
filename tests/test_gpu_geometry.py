"""The automatic geometry the decode calls take (decode_plan, num_splits = 0)
against the split rules it starts from: the power-of-two tiles rule as is, and
for the paged path the wave rule with its chunk moved to the nearer multiple of
one round of the paged kernel's CTA (4 warps x 32 positions for an int8 or
e4m3fn cache with head_dim <= 128, 4 x 16 otherwise).  Needs a device for the occupancy
wave."""
import pytest

import int8_kv_cache_gb300 as K

pytestmark = pytest.mark.gpu


def _cdiv(a, b):
    return -(-a // b)


def _snapped(cap, n, rnd):
    raw = _cdiv(cap, n)
    up, dn = _cdiv(raw, rnd) * rnd, raw // rnd * rnd
    ch = dn if dn >= 128 and raw - dn < up - raw and _cdiv(cap, dn) <= 32 else up
    return _cdiv(cap, ch), ch


@pytest.mark.parametrize("cache,D,rnd", [("int8", 128, 128), ("fp8", 128, 128),
                                          ("fp16", 128, 64), ("int8", 256, 64)])
@pytest.mark.parametrize("cap,rows,Hq,Hkv", [
    (4096, 16, 16, 2), (8192, 16, 32, 8), (1039, 16, 32, 8), (4096, 1, 32, 8), (100, 4, 8, 2),
    (65536, 2, 16, 2), (3000, 3, 16, 2), (128, 1, 16, 2), (5000, 5, 8, 2),
])
def test_paged_wave_geometry(cap, rows, Hq, Hkv, cache, D, rnd):
    dt = {"int8": K.CACHE_INT8, "fp8": K.CACHE_FP8, "fp16": K.CACHE_FP16}[cache]
    ns, ch, wsb, wave = K.decode_plan(K.PATH_PAGED, dt, cap, rows, Hq, Hkv, D, K.GEOM_WAVE)
    n0, c0 = K.split_geometry(cap, rows * Hkv, wave, 16, 128, 32, K.GEOM_WAVE, 0)
    want = (n0, c0) if n0 <= 1 else _snapped(cap, n0, rnd)
    assert (ns, ch) == want
    assert 1 <= ns <= 32 and ch % 16 == 0 and ns * ch >= cap and (ns - 1) * ch < cap
    if ns > 1:
        assert ch % rnd == 0 and ch >= 128


def test_deep_context_lands_on_whole_rounds():
    # 16 sequences of cap 4096 over 2 KV heads: the rule's 15 splits of 288
    # positions become 16 splits of 256 (two 32-position steps for each of
    # the 4 warps)
    ns, ch, _, wave = K.decode_plan(K.PATH_PAGED, K.CACHE_INT8, 4096, 16, 16, 2, 128, K.GEOM_WAVE)
    n0, c0 = K.split_geometry(4096, 32, wave, 16, 128, 32, K.GEOM_WAVE, 0)
    if wave == 456:
        assert (n0, c0) == (15, 288)
        assert (ns, ch) == (16, 256)


def test_override_and_tiles_rule_are_left_alone():
    ns, ch, _, wave = K.decode_plan(K.PATH_PAGED, K.CACHE_INT8, 4096, 16, 16, 2, 128,
                                    K.GEOM_WAVE, 288)
    assert (ns, ch) == K.split_geometry(4096, 32, wave, 16, 128, 32, K.GEOM_WAVE, 288)
    ns, ch, _, wave = K.decode_plan(K.PATH_PAGED, K.CACHE_INT8, 4096, 16, 16, 2, 128,
                                    K.GEOM_POW2_TILES)
    assert (ns, ch) == K.split_geometry(4096, 32, wave, 64, 128, 32, K.GEOM_POW2_TILES, 0)
    ns, ch, _, wave = K.decode_plan(K.PATH_DSA, K.CACHE_INT8, 2000, 8, 24, 2, 256, K.GEOM_WAVE)
    assert (ns, ch) == K.split_geometry(2000, 16, wave, 16, 128, 32, K.GEOM_WAVE, 0)
