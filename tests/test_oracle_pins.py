"""Pins of the FP64 oracle to facts fixed outside the oracle itself.

Each test checks the oracle against something it cannot reproduce by retyping
its own formula: an exact-rational / 50-digit brute force (no max subtraction,
the sink taken as an extra candidate with a zero value row), closed forms,
values the pages print, and invariants of the split form.
"""
import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as W

# --------------------------------------------------------------------------
# 50-digit brute force
# --------------------------------------------------------------------------


def _dec(fr: Fraction) -> Decimal:
    return Decimal(fr.numerator) / Decimal(fr.denominator)


def _value(code, scale_kind, scale, g, d):
    """Exact rational value of one cache element (fp16 caches as is)."""
    if isinstance(code, (np.floating,)) or np.asarray(code).dtype == np.float16:
        return Fraction(float(code))
    s = scale.reshape(-1)[0] if scale_kind == W.SCALE_PER_TENSOR else scale[g, d]
    return Fraction(float(s)) * int(code)


def brute_head(q_row, rows, kc, vc, ks, vs, kind, g, sigma, sink_logit=None):
    """O[d] and lse for one query head by direct summation of exp(s_t) with
    exact rational scores (50 significant digits for exp); a sink is one more
    term exp(s_h) in the denominator with no value row."""
    getcontext().prec = 50
    D = len(q_row)
    if len(rows) == 0:
        return [Decimal(0)] * D, None
    ws, vals = [], []
    for t in rows:
        s = Fraction(sigma) * sum(Fraction(float(q_row[d])) * _value(kc[t, g, d], kind, ks, g, d)
                                  for d in range(D))
        ws.append(_dec(s).exp())
        vals.append([_value(vc[t, g, d], kind, vs, g, d) for d in range(D)])
    Z = sum(ws)
    den = Z + (_dec(Fraction(float(sink_logit))).exp() if sink_logit is not None else 0)
    O = [sum(w * _dec(v[d]) for w, v in zip(ws, vals)) / den for d in range(D)]
    return O, Z.ln()


def _close(a, b, rel=1e-12, abs_=1e-300):
    return abs(float(a) - float(b)) <= rel * abs(float(b)) + abs_


@pytest.mark.parametrize("kind", [W.SCALE_PER_TENSOR, W.SCALE_PER_CHANNEL])
@pytest.mark.parametrize("sink", [False, True])
def test_brute_force_sparse_tiny(kind, sink):
    c = W.random_sparse(seed=11 + kind + 2 * sink, S=2, Hq=4, Hkv=2, D=8, N=16, max_sel=7,
                        invalid_frac=0.3, scale_kind=kind, sink=sink)
    O, L = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, kind,
                                   c.idx, c.sigma, c.sink)
    G = 2
    for r in range(2):
        rows = [int(t) for t in c.idx[r] if 0 <= t < 16]
        for h in range(4):
            ob, lb = brute_head(c.q[r, h], rows, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                kind, h // G, c.sigma, None if c.sink is None else c.sink[h])
            for d in range(8):
                assert _close(O[r, h, d], ob[d], abs_=1e-15), (r, h, d)
            assert _close(L[r, h], lb)


def test_brute_force_paged_tiny():
    # lengths: empty, ragged, and one longer than the cap (clamped)
    c = W.random_paged(seed=5, B=3, Hq=4, Hkv=1, D=8, bs=2, max_blocks=3, lens=[0, 3, 9],
                       sink=True)
    O, L = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                                  c.block_table, c.seq_lens, c.sigma, c.sink)
    nb, bs, Hkv, D = c.k_cache.shape
    kf = c.k_cache.reshape(nb * bs, Hkv, D)
    vf = c.v_cache.reshape(nb * bs, Hkv, D)
    for b, live in enumerate([0, 3, 6]):
        # rows by walking the block table block by block (no slot formula)
        rows = []
        for j in range(3):
            for o in range(bs):
                if len(rows) < live:
                    rows.append(int(c.block_table[b, j]) * bs + o)
        for h in range(4):
            ob, lb = brute_head(c.q[b, h], rows, kf, vf, c.k_scale, c.v_scale, c.scale_kind, 0,
                                c.sigma, c.sink[h])
            for d in range(D):
                assert _close(O[b, h, d], ob[d], abs_=1e-15)
            if live == 0:
                assert L[b, h] == -math.inf and np.all(O[b, h] == 0)
            else:
                assert _close(L[b, h], lb)


# --------------------------------------------------------------------------
# closed forms and special cases
# --------------------------------------------------------------------------

def test_identical_keys_give_mean_of_values():
    c = W.random_sparse(seed=3, S=1, Hq=2, Hkv=1, D=16, N=40, max_sel=23)
    kc = c.k_codes.copy()
    kc[:] = kc[7]  # every row holds the same key
    O, L = oracle.sparse_attention(c.q, kc, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma)
    rows = c.idx[0][(c.idx[0] >= 0) & (c.idx[0] < 40)]
    vals = c.v_codes[rows, 0, :].astype(np.float64) * c.v_scale[0].astype(np.float64)
    mean = vals.mean(axis=0)
    np.testing.assert_allclose(O[0, 0], mean, rtol=1e-12, atol=1e-14)
    s = c.sigma * float(np.dot(c.q[0, 0].astype(np.float64),
                               kc[7, 0].astype(np.float64) * c.k_scale[0].astype(np.float64)))
    assert L[0, 0] == pytest.approx(s + math.log(len(rows)), rel=1e-13, abs=1e-13)


def test_dominant_logit_gives_its_value_row():
    D = 16
    q = np.zeros(D); q[0] = 1.0
    kA = np.zeros(D, np.int8); kA[0] = 100
    kB = np.zeros(D, np.int8)
    vA = np.arange(D, dtype=np.int8) - 5
    vB = np.full(D, 77, np.int8)
    # score gap 100 * 0.5 = 50 nats
    c = W.two_candidate(q, kA, kB, vA, vB, k_scale=0.5, v_scale=0.25, sigma=1.0)
    O, L = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma)
    np.testing.assert_allclose(O[0, 0], vA.astype(np.float64) * 0.25, rtol=1e-12, atol=1e-12)


def test_empty_and_all_invalid_rows():
    c = W.random_sparse(seed=4, S=2, Hq=4, Hkv=2, D=8, N=10, max_sel=5, sink=True)
    c.idx[0, :] = -1
    c.idx[1, :] = [10, 11, -3, 99, -1]
    O, L = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma, c.sink)
    assert np.all(O == 0) and np.all(L == -math.inf)


def test_invalid_entries_are_skipped_and_duplicates_kept():
    c = W.random_sparse(seed=6, S=1, Hq=2, Hkv=1, D=8, N=30, max_sel=9)
    base = c.idx.copy()
    base[0, :] = [3, 9, 4, -1, -1, -1, -1, -1, -1]
    noisy = c.idx.copy()
    noisy[0, :] = [-5, 3, 30, 9, -1, 4, 1000, -1, -2]
    a = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                base, c.sigma)
    b = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                noisy, c.sigma)
    np.testing.assert_array_equal(a[0], b[0])
    # a duplicated candidate counts twice: same as adding ln 2 to its logit
    dup = base.copy()
    dup[0, 3] = 9
    o_dup, l_dup = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                           c.scale_kind, dup, c.sigma)
    K = c.k_codes[[3, 9, 4], 0].astype(np.float64) * c.k_scale[0]
    V = c.v_codes[[3, 9, 4], 0].astype(np.float64) * c.v_scale[0]
    for h in range(2):
        s = c.sigma * (K @ c.q[0, h].astype(np.float64))
        s[1] += math.log(2.0)
        w = np.exp(s - s.max())
        np.testing.assert_allclose(o_dup[0, h], (w @ V) / w.sum(), rtol=1e-12, atol=1e-14)


def test_per_tensor_equals_per_channel_with_constant_scales():
    c = W.random_sparse(seed=8, S=2, Hq=6, Hkv=2, D=16, N=50, max_sel=20,
                        scale_kind=W.SCALE_PER_TENSOR)
    ks_c = np.full((2, 16), c.k_scale[0], np.float32)
    vs_c = np.full((2, 16), c.v_scale[0], np.float32)
    a = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                W.SCALE_PER_TENSOR, c.idx, c.sigma)
    b = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, ks_c, vs_c, W.SCALE_PER_CHANNEL,
                                c.idx, c.sigma)
    np.testing.assert_array_equal(a[0], b[0])


def test_gqa_head_mapping_contiguous_groups():
    # Hq=6, Hkv=2: heads 0-2 read kv head 0, heads 3-5 read kv head 1.  Zeroing
    # kv head 1's values must leave heads 0-2 unchanged and zero heads 3-5.
    c = W.random_sparse(seed=9, S=1, Hq=6, Hkv=2, D=8, N=20, max_sel=10)
    vc = c.v_codes.copy()
    vc[:, 1, :] = 0
    a, _ = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma)
    b, _ = oracle.sparse_attention(c.q, c.k_codes, vc, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma)
    np.testing.assert_array_equal(a[0, :3], b[0, :3])
    assert np.all(b[0, 3:] == 0) and np.any(a[0, 3:] != 0)


# --------------------------------------------------------------------------
# the values the pages print (tests/golden/numerics_examples.json)
# --------------------------------------------------------------------------

def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, "numerics_examples.json")) as f:
        cases = {c["name"]: c for c in json.load(f)["cases"]}
    return cases[name]


def _run(c):
    return oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma)


@pytest.mark.parametrize("spread", [False, True])
def test_signed_cancellation_pin(golden_dir, spread):
    g = _golden(golden_dir, "signed value cancellation")
    O, _ = _run(W.signed_cancellation_case(spread=spread))
    # exact answer 4064 * tanh(delta/2) with delta the fp32 key scale; the page's
    # 127/256 holds to the fp32 rounding of that scale
    assert abs(O[0, 0, 0] - g["printed"]) < 1e-7
    assert np.all(O[0, :, 1:] == 0)


@pytest.mark.parametrize("sigma,name", [(1.0, "large common logit, scale 1"),
                                        (1.0 / 16.0, "large common logit, scale 1/16")])
def test_large_common_logit_pin(golden_dir, sigma, name):
    g = _golden(golden_dir, name)
    O, L = _run(W.large_common_logit_case(sigma))
    assert abs(O[0, 0, 0] - g["printed"]) <= g["abs_tol"]
    # closed form: the output is the logistic of the scaled gap 0.5 * sigma
    assert O[0, 0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-0.5 * sigma)), rel=1e-12)
    assert L[0, 0] == pytest.approx(8290560.0 * sigma + math.log1p(math.exp(0.5 * sigma)),
                                    rel=1e-15)


def test_tiny_probability_pin(golden_dir):
    g = _golden(golden_dir, "tiny probability with value_scale 2^60")
    O, _ = _run(W.tiny_probability_case(480.0, 1, 2.0 ** 60))
    assert abs(O[0, 0, 0] - g["printed"]) <= g["abs_tol"]


@pytest.mark.parametrize("q0,code,vs,gap", [(288.0, 100, 2.0 ** 16, 18.0),
                                            (320.0, 1, 2.0 ** 28, 20.0),
                                            (480.0, 1, 2.0 ** 60, 30.0)])
def test_tiny_probability_closed_forms(q0, code, vs, gap):
    O, L = _run(W.tiny_probability_case(q0, code, vs))
    want = code * vs * math.exp(-gap) / (1.0 + math.exp(-gap))
    assert O[0, 0, 0] == pytest.approx(want, rel=1e-12)
    assert L[0, 0] == pytest.approx(math.log1p(math.exp(-gap)), rel=1e-12)


# --------------------------------------------------------------------------
# split form and the combine
# --------------------------------------------------------------------------

def test_combine_of_any_partition_equals_whole():
    rng = np.random.default_rng(21)
    D = 12
    for trial in range(40):
        T = int(rng.integers(1, 40))
        K = rng.standard_normal((T, D)) * 3
        V = rng.standard_normal((T, D))
        q = rng.standard_normal(D)
        sig = float(rng.uniform(0.05, 1.0))
        o_whole, l_whole = oracle.attend(q, K, V, sig)
        ncut = int(rng.integers(0, 6))
        cuts = np.sort(rng.integers(0, T + 1, size=ncut))  # repeated cuts -> empty parts
        edges = [0] + list(cuts) + [T]
        parts = [oracle.partial(q, K[a:b], V[a:b], sig) for a, b in zip(edges[:-1], edges[1:])]
        if rng.random() < 0.5:
            parts.append(oracle.partial(q, K[:0], V[:0], sig))  # an extra empty split
            parts = parts[::-1]
        o, lse = oracle.combine([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts])
        np.testing.assert_allclose(o, o_whole, rtol=1e-12, atol=1e-13)
        assert lse == pytest.approx(l_whole, rel=1e-13, abs=1e-13)


def test_single_split_equals_unsplit():
    rng = np.random.default_rng(3)
    K = rng.standard_normal((17, 8)); V = rng.standard_normal((17, 8)); q = rng.standard_normal(8)
    m, l, a = oracle.partial(q, K, V, 0.3)
    o, lse = oracle.combine([m], [l], [a], s_h=0.7)
    o2, lse2 = oracle.attend(q, K, V, 0.3)
    np.testing.assert_allclose(o, oracle.apply_head_sink(o2, lse2, 0.7), rtol=1e-14, atol=1e-15)
    assert lse == pytest.approx(lse2, rel=1e-15)


@pytest.mark.parametrize("chunk", [1, 3, 4, 7, 64])
def test_sparse_split_form_matches_whole(chunk):
    c = W.random_sparse(seed=30 + chunk, S=3, Hq=4, Hkv=2, D=8, N=64, max_sel=21,
                        invalid_frac=0.25, sink=True)
    ns = -(-21 // chunk)
    m, l, a = oracle.sparse_split_partials(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                           c.scale_kind, c.idx, c.sigma, ns, chunk)
    O, L = oracle.combine_all(m, l, a, c.sink)
    O2, L2 = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                     c.scale_kind, c.idx, c.sigma, c.sink)
    np.testing.assert_allclose(O, O2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L, L2, rtol=1e-13)


@pytest.mark.parametrize("ns,tile,G", [(1, 8, 4), (2, 8, 4), (3, 8, 4), (5, 8, 4), (4, 3, 1),
                                       (7, 6, 2)])
def test_prefill_block_split_form_matches_whole(ns, tile, G):
    # the split prefill's ranges (small tiles and 8-position blocks so that
    # tiles straddle rows and splits get one block, several or none) cover
    # [0, N) once per tile, and the merge of the partials is the whole
    Hkv = 2
    c = W.random_sparse(seed=40 + ns + tile, S=7, Hq=G * Hkv, Hkv=Hkv, D=8, N=61, max_sel=19,
                        invalid_frac=0.2, sink=True)
    c.idx[3, 5] = c.idx[3, 2]  # a repeated entry counts twice in its split
    c.idx[5, :] = -1            # a row with nothing
    for ranges in oracle.prefill_block_ranges(c.idx, 61, G, ns, tile=tile, block=8):
        assert len(ranges) == ns and ranges[0][0] == 0 and ranges[-1][1] == 61
        assert all(ranges[k][1] == ranges[k + 1][0] for k in range(ns - 1))
        assert all(lo <= hi for lo, hi in ranges)
    m, l, a = oracle.prefill_split_partials(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                            c.scale_kind, c.idx, c.sigma, ns, tile=tile,
                                            block=8)
    O, L = oracle.combine_all(m, l, a, c.sink)
    O2, L2 = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                     c.scale_kind, c.idx, c.sigma, c.sink)
    np.testing.assert_allclose(O, O2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L, L2, rtol=1e-13)
    assert np.all(np.isneginf(m[5])) and np.all(l[5] == 0)


def test_prefill_block_ranges_by_hand():
    # one tile (G = 2, three rows), 8-position blocks: the rows' candidates sit
    # in blocks 0, 2, 3 and 6, so 3 splits take ranks [0, 1), [1, 2), [2, 4)
    idx = np.array([[1, 17, -1], [20, 25, 99], [50, 3, 18]], np.int32)
    (ranges,) = oracle.prefill_block_ranges(idx, 60, 2, 3, tile=8, block=8)
    assert ranges == [(0, 16), (16, 24), (24, 60)]
    # more splits than blocks: ranks [0,0) [0,1) [1,2) [2,2) [2,3) [3,4); the
    # splits with no rank get empty ranges
    (ranges,) = oracle.prefill_block_ranges(idx, 60, 2, 6, tile=8, block=8)
    assert ranges == [(0, 0), (0, 16), (16, 24), (24, 24), (24, 48), (48, 60)]
    # no candidate at all: every range empty but the last, which is [0, N)
    (ranges,) = oracle.prefill_block_ranges(np.full((3, 3), -1, np.int32), 60, 2, 3, tile=8,
                                            block=8)
    assert ranges == [(0, 0), (0, 0), (0, 60)]


@pytest.mark.parametrize("chunk,ns", [(2, 12), (4, 6), (16, 2), (32, 1), (4, 9)])
def test_paged_split_form_matches_whole(chunk, ns):
    c = W.random_paged(seed=7, B=4, Hq=4, Hkv=2, D=8, bs=2, max_blocks=12, lens=[0, 5, 24, 30],
                       sink=True)
    m, l, a = oracle.paged_split_partials(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                          c.scale_kind, c.block_table, c.seq_lens, c.sigma, ns,
                                          chunk)
    O, L = oracle.combine_all(m, l, a, c.sink)
    O2, L2 = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                    c.scale_kind, c.block_table, c.seq_lens, c.sigma, c.sink)
    if ns * chunk >= 24:
        np.testing.assert_allclose(O, O2, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(L, L2, rtol=1e-13)
    else:
        # splits that do not reach the cap drop the tail: not equal in general
        assert ns * chunk < 24


def test_sink_post_hoc_equals_extra_candidate():
    c = W.random_sparse(seed=12, S=2, Hq=4, Hkv=1, D=8, N=25, max_sel=9, sink=True)
    O, L = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma, c.sink)
    for r in range(2):
        rows = c.idx[r][(c.idx[r] >= 0) & (c.idx[r] < 25)]
        K = c.k_codes[rows, 0].astype(np.float64) * c.k_scale[0]
        V = c.v_codes[rows, 0].astype(np.float64) * c.v_scale[0]
        for h in range(4):
            s = c.sigma * (K @ c.q[r, h].astype(np.float64))
            s_all = np.concatenate([s, [float(c.sink[h])]])
            w = np.exp(s_all - s_all.max())
            V_all = np.vstack([V, np.zeros((1, 8))])
            np.testing.assert_allclose(O[r, h], (w @ V_all) / w.sum(), rtol=1e-12, atol=1e-14)


def test_no_sink_equals_minus_infinity_sink():
    c = W.random_sparse(seed=13, S=1, Hq=4, Hkv=2, D=8, N=25, max_sel=9)
    a = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                c.idx, c.sigma, None)
    b = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                c.idx, c.sigma, np.full(4, -np.inf, np.float32))
    np.testing.assert_array_equal(a[0], b[0])


# --------------------------------------------------------------------------
# gathers
# --------------------------------------------------------------------------

def test_paged_slots_match_block_scatter():
    """Scatter a logical [B, cap] token array into the pool block by block with
    the table, then gather it back through the slot ids."""
    c = W.random_paged(seed=2, B=5, Hq=2, Hkv=1, D=4, bs=4, max_blocks=6, lens=[0, 1, 4, 17, 40])
    bs, mb = 4, 6
    cap = bs * mb
    logical = np.arange(5 * cap).reshape(5, cap) + 1000
    pool = np.full(c.k_cache.shape[0] * bs, -7, dtype=np.int64).reshape(-1, bs)
    for b in range(5):
        for j in range(mb):
            p = c.block_table[b, j]
            if p >= 0:
                pool[p] = logical[b, j * bs:(j + 1) * bs]
    slots = oracle.paged_slots(c.block_table, c.seq_lens, bs)
    flat = pool.reshape(-1)
    for b, L in enumerate([0, 1, 4, 17, 24]):
        np.testing.assert_array_equal(flat[slots[b, :L]], logical[b, :L])
        assert np.all(slots[b, L:] == -1)


def test_paged_equals_sparse_on_identity_layout():
    c = W.deep_context(seed=1, B=2, cap=64, live=37, Hq=4, Hkv=2, D=8, bs=16, sink=True)
    O, L = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                                  c.block_table, c.seq_lens, c.sigma, c.sink)
    kf = c.k_cache.reshape(-1, 2, 8)
    vf = c.v_cache.reshape(-1, 2, 8)
    for b in range(2):
        idx = (np.arange(37) + b * 64).reshape(1, -1).astype(np.int32)
        O2, L2 = oracle.sparse_attention(c.q[b:b + 1], kf, vf, c.k_scale, c.v_scale, c.scale_kind,
                                         idx, c.sigma, c.sink)
        np.testing.assert_array_equal(O[b], O2[0])
        np.testing.assert_array_equal(L[b], L2[0])


def test_fp16_cache_taken_as_is():
    c = W.deep_context(seed=4, cache="fp16", B=1, cap=32, live=20, Hq=2, Hkv=1, D=8)
    O, _ = oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale * 3, c.v_scale * 5,
                                  c.scale_kind, c.block_table, c.seq_lens, c.sigma)
    K = c.k_cache.reshape(-1, 1, 8)[:20, 0].astype(np.float64)
    V = c.v_cache.reshape(-1, 1, 8)[:20, 0].astype(np.float64)
    s = c.sigma * (K @ c.q[0, 0].astype(np.float64))
    w = np.exp(s - s.max())
    np.testing.assert_allclose(O[0, 0], (w @ V) / w.sum(), rtol=1e-12)


def test_query_folding_case_closed_form():
    # logits sigma * (32768 * 8 - 32766 * 8) = 16 and 0, values 1 and 0
    c = W.query_folding_case()
    O, L = oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma)
    assert O[0, 0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-16.0)), rel=1e-15)
    assert L[0, 0] == pytest.approx(16.0 + math.log1p(math.exp(-16.0)), rel=1e-15)
    assert np.all(O[0, :, 1:] == 0)
