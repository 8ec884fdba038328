"""Pins of the quantize-on-write oracle: closed-form properties of symmetric
rounding, exact ties, saturation, NaN handling and the slot scatter."""
import numpy as np

import oracle


def test_round_half_to_even_on_exact_ties():
    # scale 1 (a power of two): x / scale is exact, so ties are ties
    x = np.array([[0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 126.5]], np.float16)
    got = oracle.quantize_rows(x, np.array([1.0], np.float32), oracle.SCALE_PER_TENSOR, 0)
    np.testing.assert_array_equal(got[0], [0, 2, 2, 0, -2, -2, 4, 126])


def test_saturation_and_nan():
    x = np.array([[1000.0, -1000.0, 127.0, -127.0, 127.6, np.nan, np.inf, -np.inf]], np.float16)
    got = oracle.quantize_rows(x, np.array([1.0], np.float32), oracle.SCALE_PER_TENSOR, 0)
    np.testing.assert_array_equal(got[0], [127, -127, 127, -127, 127, 0, 127, -127])


def test_round_trip_error_is_at_most_half_a_step():
    rng = np.random.default_rng(0)
    scale = np.exp(rng.uniform(-6, 2, size=(3, 64))).astype(np.float32)
    x = (rng.uniform(-127, 127, size=(50, 3, 64)) * scale).astype(np.float16)
    for g in range(3):
        codes = oracle.quantize_rows(x[:, g], scale, oracle.SCALE_PER_CHANNEL, g)
        back = codes.astype(np.float64) * scale[g].astype(np.float64)
        err = np.abs(back - x[:, g].astype(np.float64))
        # half a step, plus the fp32 rounding of the quotient at a tie
        assert np.all(err <= 0.5 * scale[g] * (1 + 1e-6) + 1e-30)


def test_per_tensor_equals_per_channel_with_constant_scale():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((20, 2, 16)) * 3).astype(np.float16)
    a = oracle.quantize_rows(x[:, 1], np.array([0.037], np.float32), oracle.SCALE_PER_TENSOR, 1)
    b = oracle.quantize_rows(x[:, 1], np.full((2, 16), 0.037, np.float32),
                             oracle.SCALE_PER_CHANNEL, 1)
    np.testing.assert_array_equal(a, b)


def test_slot_scatter_writes_exactly_the_mapped_rows():
    rng = np.random.default_rng(2)
    nb, bs, Hkv, D = 5, 16, 2, 8
    kc = rng.integers(-100, 100, size=(nb, bs, Hkv, D)).astype(np.int8)
    vc = rng.integers(-100, 100, size=(nb, bs, Hkv, D)).astype(np.int8)
    T = 7
    kn = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    vn = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    slots = np.array([3, -1, 79, 16, 80, 0, -5], np.int32)  # 80 is past the pool: skipped
    ks = np.array([0.02], np.float32)
    vs = np.array([0.03], np.float32)
    k2, v2 = oracle.reshape_and_cache(kn, vn, slots, kc, vc, ks, vs, oracle.SCALE_PER_TENSOR)
    flat_k, flat_v = k2.reshape(-1, Hkv, D), v2.reshape(-1, Hkv, D)
    touched = {3: 0, 79: 2, 16: 3, 0: 5}
    for s in range(nb * bs):
        if s in touched:
            n = touched[s]
            for g in range(Hkv):
                np.testing.assert_array_equal(
                    flat_k[s, g], np.clip(np.rint(kn[n, g].astype(np.float32) / np.float32(0.02)),
                                          -127, 127).astype(np.int8))
        else:
            np.testing.assert_array_equal(flat_k[s], kc.reshape(-1, Hkv, D)[s])
            np.testing.assert_array_equal(flat_v[s], vc.reshape(-1, Hkv, D)[s])
