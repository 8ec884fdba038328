"""Pins of the oracle's float8 e4m3fn cache codec.

[onnxruntime PR 29912, Schema: the cache element type is one of float16,
bfloat16, int8, float8e4m3fn; the quantised paths dequantise with k_scale /
v_scale, PER_TENSOR or PER_CHANNEL.]  The oracle decodes e4m3fn bit patterns
from the format's definition and encodes by rounding to nearest even with
saturation.  Pinned against PyTorch's own float8_e4m3fn dtype (an independent
implementation), the format's landmark values, and exhaustive midpoints.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_decoder_exhaustive_against_torch():
    ref = _torch_decode(np.arange(256))
    got = np.array([oracle.e4m3fn_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def test_decoder_landmarks():
    v = oracle.e4m3fn_value
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0          # largest finite
    assert v(0x01) == 2.0 ** -9                            # smallest subnormal
    assert v(0x07) == 7 * 2.0 ** -9                        # largest subnormal
    assert v(0x08) == 2.0 ** -6                            # smallest normal
    assert v(0x38) == 1.0 and v(0xB8) == -1.0
    assert v(0x39) == 1.125                                # 1 + 1/8
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))     # the only NaNs
    assert v(0x00) == 0.0 and math.copysign(1.0, v(0x80)) == -1.0
    assert sum(math.isnan(v(c)) for c in range(256)) == 2  # no infinities


def test_encoder_matches_torch_in_range():
    rng = np.random.default_rng(0)
    # log-uniform magnitudes from deep subnormal to just below the largest
    # finite value, both signs
    mag = np.exp2(rng.uniform(-14.0, math.log2(448.0), size=200000))
    x = (mag * rng.choice([-1.0, 1.0], size=mag.shape)).astype(np.float32)
    got = np.array([oracle.e4m3fn_encode(float(a)) for a in x], dtype=np.uint8)
    np.testing.assert_array_equal(got, _torch_encode(x))


def test_encoder_midpoints_round_to_even():
    vals = np.array([oracle.e4m3fn_value(c) for c in range(0x7F)])  # 0 .. 448, ascending
    assert np.all(np.diff(vals) > 0)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)  # exact in fp32
    got = np.array([oracle.e4m3fn_encode(float(m)) for m in mids])
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)   # the even mantissa of the two neighbours
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(got, _torch_encode(mids))
    neg = np.array([oracle.e4m3fn_encode(-float(m)) for m in mids])
    np.testing.assert_array_equal(neg, want | 0x80)


def test_encoder_round_trip_saturation_and_nan():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3fn_encode(oracle.e4m3fn_value(c)) == c
    # readings: beyond the largest finite value saturates (torch gives NaN
    # there), NaN stores 0, a value rounding to zero keeps its sign
    assert oracle.e4m3fn_encode(463.99) == 0x7E and oracle.e4m3fn_encode(1e30) == 0x7E
    assert oracle.e4m3fn_encode(-1e30) == 0xFE and oracle.e4m3fn_encode(math.inf) == 0x7E
    assert oracle.e4m3fn_encode(math.nan) == 0x00
    assert oracle.e4m3fn_encode(2.0 ** -11) == 0x00       # a quarter of the smallest subnormal
    assert oracle.e4m3fn_encode(-(2.0 ** -11)) == 0x80
    assert oracle.e4m3fn_encode(2.0 ** -10) == 0x00       # half of it: the tie goes to even 0
    assert oracle.e4m3fn_encode(3 * 2.0 ** -10) == 0x02   # 1.5 ulp: the tie goes to even 2


def test_fp8_cache_equals_fp16_cache_of_its_values():
    # with unit scales an fp8 cache holds exactly the fp16 values it decodes to
    c = W.random_paged(seed=2, B=3, Hq=8, Hkv=2, D=32, bs=16, max_blocks=4, lens=[50, 1, 64],
                       cache="fp8", sink=True)
    c.k_scale = np.ones_like(c.k_scale)
    c.v_scale = np.ones_like(c.v_scale)
    a = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                               c.block_table, c.seq_lens, c.sigma, c.sink)
    kf = _torch_decode(c.k_cache).astype(np.float16)
    vf = _torch_decode(c.v_cache).astype(np.float16)
    b = oracle.paged_attention(c.q, kf, vf, c.k_scale, c.v_scale, c.scale_kind, c.block_table,
                               c.seq_lens, c.sigma, c.sink)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_fp8_dequantize_scales_decoded_values():
    codes = np.array([[0x38, 0xB8, 0x7E, 0x01]], dtype=np.uint8)   # 1, -1, 448, 2^-9
    ks = np.array([[0.5, 2.0, 0.25, 8.0]], dtype=np.float32)
    got = oracle.dequantize(codes, ks, W.SCALE_PER_CHANNEL, 0)
    np.testing.assert_array_equal(got, [[0.5, -2.0, 112.0, 2.0 ** -6]])
    got = oracle.dequantize(codes, np.array([4.0], np.float32), W.SCALE_PER_TENSOR, 0)
    np.testing.assert_array_equal(got, [[4.0, -4.0, 1792.0, 2.0 ** -7]])


@pytest.mark.parametrize("kind", [W.SCALE_PER_TENSOR, W.SCALE_PER_CHANNEL])
def test_fp8_quantize_on_write_rows(kind):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((6, 2, 16)) * 3).astype(np.float16)
    if kind == W.SCALE_PER_TENSOR:
        s = np.array([0.01], np.float32)
    else:
        s = np.exp(rng.uniform(-5, -3, size=(2, 16))).astype(np.float32)
    for g in range(2):
        got = oracle.quantize_rows_fp8(x[:, g], s, kind, g)
        q = x[:, g].astype(np.float32) / (s[0] if kind == W.SCALE_PER_TENSOR else s[g])
        sat = np.abs(q) > 448
        want = _torch_encode(q)
        want[sat] = np.where(q[sat] > 0, 0x7E, 0xFE)  # torch gives NaN beyond 448
        np.testing.assert_array_equal(got, want)
