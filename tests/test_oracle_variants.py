"""Pins of the oracle's paged-decode variants: softcap and sliding window.

[onnxruntime PR 29912 "PagedAttention: quantized KV cache ...", CUDA kernels:
the paged decode kernel has native head-sink, softcap, sliding-window and
on-the-fly dequantisation.]  The pages name both options without defining
them; the oracle takes softcap c as s -> c * tanh(s / c) on the scaled score
and a window w as the positions [L - 1 - w, L) of a decode query at L - 1.
These tests pin those readings to facts computed another way: a 50-digit
brute force with tanh written from exponentials, closed forms (a logistic
value, tanh(ln 3 / 2) = 1/2), limits, and hand-written slot tables.
"""
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as W


def _dec(x) -> Decimal:
    fr = Fraction(x)
    return Decimal(fr.numerator) / Decimal(fr.denominator)


def _tanh_dec(x: Decimal) -> Decimal:
    e = (2 * x).exp()
    return (e - 1) / (e + 1)


def _brute(q_row, rows, kf, vf, ks, vs, kind, g, sigma, softcap, sink_logit=None):
    """O[d], lse of one head by direct summation (no max subtraction), scores
    exact rationals, the cap and exp in 50 digits, the sink one more term."""
    getcontext().prec = 50
    D = len(q_row)
    if not rows:
        return [Decimal(0)] * D, None

    def val(code, scale, d):
        s = scale.reshape(-1)[0] if kind == W.SCALE_PER_TENSOR else scale[g, d]
        return Fraction(float(s)) * int(code)

    ws, vals = [], []
    for t in rows:
        s = _dec(Fraction(sigma) * sum(Fraction(float(q_row[d])) * val(kf[t, g, d], ks, d)
                                       for d in range(D)))
        if softcap > 0:
            c = _dec(softcap)
            s = c * _tanh_dec(s / c)
        ws.append(s.exp())
        vals.append([val(vf[t, g, d], vs, d) for d in range(D)])
    Z = sum(ws)
    den = Z + (_dec(float(sink_logit)).exp() if sink_logit is not None else 0)
    return [sum(w * _dec(v[d]) for w, v in zip(ws, vals)) / den for d in range(D)], Z.ln()


def _close(a, b, rel=1e-12, abs_=1e-15):
    return abs(float(a) - float(b)) <= rel * abs(float(b)) + abs_


@pytest.mark.parametrize("softcap,window", [(0.0, 2), (4.0, -1), (2.5, 3), (1.0, 0)])
def test_brute_force_paged_variants(softcap, window):
    lens = [0, 1, 5, 9]          # empty, one token, ragged, clamped to the cap 6
    c = W.random_paged(seed=21, B=4, Hq=4, Hkv=2, D=8, bs=2, max_blocks=3, lens=lens, sink=True)
    c.sigma = 0.7                # scores of a few units, so the cap bends them
    O, L = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                                  c.block_table, c.seq_lens, c.sigma, c.sink, softcap=softcap,
                                  window=window)
    nb, bs, Hkv, D = c.k_cache.shape
    kf = c.k_cache.reshape(nb * bs, Hkv, D)
    vf = c.v_cache.reshape(nb * bs, Hkv, D)
    for b, live in enumerate([0, 1, 5, 6]):
        # every token of the sequence by walking the block table, then keep the
        # last (window + 1) of them
        toks = [int(c.block_table[b, j]) * bs + o for j in range(3) for o in range(bs)][:live]
        if window >= 0:
            toks = toks[-(window + 1):] if live else []
        for h in range(4):
            ob, lb = _brute(c.q[b, h], toks, kf, vf, c.k_scale, c.v_scale, c.scale_kind, h // 2,
                            c.sigma, softcap, c.sink[h])
            for d in range(D):
                assert _close(O[b, h, d], ob[d]), (b, h, d)
            if not toks:
                assert L[b, h] == -math.inf and np.all(O[b, h] == 0)
            else:
                assert _close(L[b, h], lb)


def test_softcap_saturates_to_logistic():
    # scores 1000 and 0 under cap 5: capped to 5 (tanh(200) = 1 in fp64) and 0,
    # so the weight of the first value row is the logistic 1 / (1 + e^-5)
    K = np.array([[1000.0], [0.0]])
    V = np.array([[1.0], [0.0]])
    o, lse = oracle.attend(np.array([1.0]), K, V, 1.0, softcap=5.0)
    assert o[0] == pytest.approx(1.0 / (1.0 + math.exp(-5.0)), rel=1e-15)
    assert lse == pytest.approx(math.log(math.exp(5.0) + 1.0), rel=1e-15)


def test_softcap_at_half_tanh():
    # tanh(ln(3)/2) = 1/2 exactly, so a score of c*ln(3)/2 is capped to c/2;
    # the score is sigma * q * k with sigma = 1/16 (the cap acts after sigma)
    c = 10.0
    k = c * math.log(3.0) / 2.0 * 16.0
    o, lse = oracle.attend(np.array([1.0]), np.array([[k], [0.0]]), np.array([[1.0], [0.0]]),
                           1.0 / 16.0, softcap=c)
    assert o[0] == pytest.approx(math.exp(5.0) / (math.exp(5.0) + 1.0), rel=1e-14)
    assert lse == pytest.approx(math.log(math.exp(5.0) + 1.0), rel=1e-14)


def test_softcap_large_cap_is_uncapped():
    c = W.random_paged(seed=3, B=2, Hq=4, Hkv=1, D=16, bs=16, max_blocks=4, lens=[40, 64])
    a = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                               c.block_table, c.seq_lens, c.sigma)
    b = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                               c.block_table, c.seq_lens, c.sigma, softcap=1e7)
    # c tanh(s/c) = s - s^3 / (3 c^2) + ...: |s| < 10 gives < 4e-13
    np.testing.assert_allclose(b[0], a[0], rtol=0, atol=1e-11)
    np.testing.assert_allclose(b[1], a[1], rtol=0, atol=1e-11)


def test_window_zero_is_the_last_token_and_wide_window_is_off():
    c = W.random_paged(seed=4, B=3, Hq=4, Hkv=2, D=16, bs=16, max_blocks=4, lens=[1, 33, 64],
                       sink=False)
    O0, L0 = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                    c.scale_kind, c.block_table, c.seq_lens, c.sigma, window=0)
    nb, bs, Hkv, D = c.k_cache.shape
    for b, live in enumerate([1, 33, 64]):
        t = live - 1
        slot = int(c.block_table[b, t // bs]) * bs + t % bs
        for h in range(4):
            g = h // 2
            v = c.v_cache.reshape(-1, Hkv, D)[slot, g].astype(np.float64) * c.v_scale[g]
            np.testing.assert_allclose(O0[b, h], v, rtol=1e-15, atol=0)
    full = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                                  c.block_table, c.seq_lens, c.sigma)
    for w in (63, 64, 1000):
        wide = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                      c.scale_kind, c.block_table, c.seq_lens, c.sigma, window=w)
        np.testing.assert_array_equal(wide[0], full[0])
        np.testing.assert_array_equal(wide[1], full[1])


def test_windowed_slots_by_hand():
    # bs 2, blocks [5, 2, 7]: positions 0..5 sit in rows 10 11 | 4 5 | 14 15.
    bt = np.array([[5, 2, 7], [5, 2, 7]])
    s = oracle.paged_slots(bt, np.array([5, 6]), 2, window=2)
    np.testing.assert_array_equal(s, [[-1, -1, 4, 5, 14, -1], [-1, -1, -1, 5, 14, 15]])
    s = oracle.paged_slots(bt, np.array([2, 0]), 2, window=5)
    np.testing.assert_array_equal(s, [[10, 11, -1, -1, -1, -1], [-1] * 6])


@pytest.mark.parametrize("window", [0, 1, 15, 16, 17, 40, 200])
def test_window_chunks_cover_the_window_once(window):
    cap = 96
    span = oracle.window_span(cap, window)
    for chunk in (16, 32, 64):
        ns = -(-span // chunk)
        if ns > 32:
            continue
        for L in range(cap + 1):
            got = []
            for lo, hi in oracle.window_chunk_bounds(L, window, chunk, ns):
                assert lo <= hi
                got.extend(range(lo, hi))
            assert got == list(range(oracle.window_start(L, window), L)), (L, chunk)


@pytest.mark.parametrize("window,softcap", [(-1, 3.0), (20, 0.0), (37, 2.0)])
def test_windowed_split_partials_combine_to_the_whole(window, softcap):
    c = W.random_paged(seed=8, B=3, Hq=8, Hkv=2, D=16, bs=16, max_blocks=6, lens=[0, 50, 96],
                       sink=True)
    c.sigma = 0.5
    O, L = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                                  c.block_table, c.seq_lens, c.sigma, c.sink, softcap=softcap,
                                  window=window)
    span = oracle.window_span(96, window)
    for chunk in (16, 48):
        ns = -(-span // chunk)
        m, l, a = oracle.paged_split_partials(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                              c.scale_kind, c.block_table, c.seq_lens, c.sigma,
                                              ns, chunk, softcap=softcap, window=window)
        Oc, Lc = oracle.combine_all(m, l, a, c.sink)
        np.testing.assert_allclose(Oc, O, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(Lc, L, rtol=1e-12, atol=0)
