"""The numerical-eligibility checks and the FP32 path, against the FP64 oracle.

[onnxruntime PR 33707, Summary of Changes §1 and the review cases: a CTA
evaluates its heads in FP32 on the CUDA cores when an element of Q * k_scale is
not finite or beyond 65504, when a head's bound on the logit shift from
rounding Q' exceeds 0.125 nats, when a value scale is not finite, or when some
|value_scale| > 2^16 and a valid candidate is more than 20 nats below the
running maximum; the FP32 path shifts terms more than 80 nats down by 2^80.]
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_close_oracle, assert_lse_close, lse_bound, oracle_dsa, oracle_paged,
                     paged_to_device, run_dsa, run_paged)

pytestmark = pytest.mark.gpu

FP32_PATH = 0x10


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()
    return K


def _flags():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _ws_layout(m, l, a, R, Hkv, G, ns, D):
    """Oracle partials [R, Hq, ns(, D)] -> workspace layout [R*Hkv, ns, G(, D)]."""
    m = m.reshape(R, Hkv, G, ns).transpose(0, 1, 3, 2).reshape(R * Hkv, ns, G)
    l = l.reshape(R, Hkv, G, ns).transpose(0, 1, 3, 2).reshape(R * Hkv, ns, G)
    a = a.reshape(R, Hkv, G, ns, D).transpose(0, 1, 3, 2, 4).reshape(R * Hkv, ns, G, D)
    return m, l, a


@pytest.mark.parametrize("spread", [False, True])
def test_query_folding_rounding_takes_the_fp32_path(K, spread):
    c = W.query_folding_case(spread=spread)
    want = 1.0 / (1.0 + math.exp(-16.0))  # fp16 rounding of Q' would give 0.5
    for kw in (dict(num_splits=1, chunk=192), dict(num_splits=3, chunk=64), dict(prefill=True),
               dict(prefill=True, staged=True, num_splits=3)):
        f = _flags()
        o, l = run_dsa(c, flags=f, **kw)
        assert abs(o[0, 0, 0] - want) <= 2e-3, (kw, o[0, 0, 0])
        assert abs(l[0, 0] - 16.0) <= 1e-5 + 1e-6 * 16, (kw, l[0, 0])
        assert int(f.item()) & FP32_PATH, kw


@pytest.mark.parametrize("S,Hq,max_sel", [(2, 8, 300), (3, 24, 509), (1, 32, 64)])
def test_large_queries_dsa(K, S, Hq, max_sel):
    c = W.random_sparse(seed=S + Hq, S=S, Hq=Hq, Hkv=2, D=256, N=1000, max_sel=max_sel,
                        invalid_frac=0.1, sink=True)
    c.q = (c.q.astype(np.float32) * 32).astype(np.float16)  # every head over the budget
    ref_o, ref_l = oracle_dsa(c)
    for kw in (dict(), dict(num_splits=1, chunk=512), dict(num_splits=-(-max_sel // 64), chunk=64),
               dict(prefill=True), dict(prefill=True, staged=True, num_splits=4)):
        f = _flags()
        o, l = run_dsa(c, flags=f, **kw)
        assert_close_oracle(o, ref_o, f"{kw}")
        assert_lse_close(l, ref_l, 1e-4)
        assert int(f.item()) & FP32_PATH


@pytest.mark.parametrize("cache", ["int8", "fp8"])
@pytest.mark.parametrize("softcap,window", [(0.0, -1), (2.0, 100)])
def test_large_queries_paged(K, cache, softcap, window):
    c = W.random_paged(seed=90, B=5, Hq=16, Hkv=4, D=128, bs=16, max_blocks=32,
                       lens=[0, 3, 200, 512, 900], sink=True, cache=cache)
    c.q = (c.q.astype(np.float32) * 64).astype(np.float16)
    ref_o, ref_l = oracle_paged(c, softcap, window)
    d = paged_to_device(c)
    for ns, ch in [(0, 0), (1, 512), (4, 128)]:
        if ns and ns * ch < K.window_span(512, window):
            continue
        f = _flags()
        o, l = run_paged(c, d, num_splits=ns, chunk=ch, flags=f, softcap=softcap, window=window)
        assert_close_oracle(o, ref_o, f"{cache} ns {ns}")
        assert_lse_close(l, ref_l, 1e-4)
        assert int(f.item()) & FP32_PATH
    m, l, a = run_paged(c, d, num_splits=4, chunk=128, softcap=softcap, window=window,
                        partials=True)
    rm, rl, ra = oracle.paged_split_partials(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                             c.scale_kind, c.block_table, c.seq_lens, c.sigma,
                                             4, 128, softcap=softcap, window=window)
    rm, rl, ra = _ws_layout(rm, rl, ra, 5, 4, 4, 4, 128)
    live = np.isfinite(rm)
    assert np.array_equal(np.isfinite(m), live)
    np.testing.assert_allclose(m[live], rm[live], rtol=1e-6, atol=1e-5)
    np.testing.assert_allclose(l[live], rl[live], rtol=1e-4)
    np.testing.assert_allclose(a[live], ra[live], rtol=1e-4, atol=1e-4 * np.abs(ra).max())


def test_tiny_probability_value_scale_2_60(K):
    """p = e^-30 on a value scale of 2^60: the fp16 tile would drop the term; the
    partial (an FP32 number) and the lse keep it (the fp16 output overflows)."""
    c = W.tiny_probability_case(480.0, 1, 2.0 ** 60)
    rm, rl, ra = oracle.sparse_split_partials(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                              c.scale_kind, c.idx, c.sigma, 3, 64)
    rm, rl, ra = _ws_layout(rm, rl, ra, 1, 1, 4, 3, 64)
    f = _flags()
    m, l, a = run_dsa(c, num_splits=3, chunk=64, partials=True, flags=f)
    assert int(f.item()) & FP32_PATH
    live = np.isfinite(rm)
    assert np.array_equal(np.isfinite(m), live)
    np.testing.assert_allclose(m[live], rm[live], atol=1e-6)
    np.testing.assert_allclose(l[live], rl[live], rtol=1e-6)
    np.testing.assert_allclose(a[live], ra[live], rtol=1e-5, atol=1e-3)
    assert abs(a[0, 0, 0, 0] - 107886.0475) < 1.0
    _, ref_l = oracle_dsa(c)
    for kw in (dict(num_splits=1, chunk=192), dict(prefill=True)):
        _, lse = run_dsa(c, **kw)
        assert_lse_close(lse, ref_l, 1e-5)


@pytest.mark.parametrize("q0,vs,gap,fp32", [(320.0, 2.0 ** 28, 20.0, False),
                                            (336.0, 2.0 ** 28, 21.0, True),
                                            (352.0, 2.0 ** 16, 22.0, False)])
def test_tail_depth_threshold(K, q0, vs, gap, fp32):
    """A candidate exactly 20 nats down, or a value scale of exactly 2^16, stays
    on the tensor cores; 21 nats down with 2^28 goes to the FP32 path."""
    c = W.tiny_probability_case(q0, 1, vs)
    want = vs * math.exp(-gap) / (1 + math.exp(-gap))
    f = _flags()
    o, _ = run_dsa(c, num_splits=1, chunk=192, flags=f)
    assert bool(int(f.item()) & FP32_PATH) == fp32
    if fp32 or vs <= 2.0 ** 16:
        assert abs(o[0, 0, 0] - want) <= 2e-3 + 1e-2 * want, (o[0, 0, 0], want)


def test_large_value_scales_with_deep_candidates(K):
    """|value_scale| between 2^16 and 2^19 and logits spread over tens of nats:
    the CTAs with a candidate more than 20 nats down take the FP32 path; the
    partials of every CTA match the oracle."""
    c = W.random_sparse(seed=61, S=4, Hq=16, Hkv=2, D=256, N=3000, max_sel=1024,
                        invalid_frac=0.0)
    assert c.scale_kind == W.SCALE_PER_CHANNEL
    rng = np.random.default_rng(1)
    c.v_scale = np.exp2(rng.uniform(16.5, 19, size=c.v_scale.shape)).astype(np.float32)
    c.q = (c.q.astype(np.float32) * 3).astype(np.float16)
    ns, ch = 8, 128
    rm, rl, ra = oracle.sparse_split_partials(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                              c.scale_kind, c.idx, c.sigma, ns, ch)
    rm, rl, ra = _ws_layout(rm, rl, ra, 4, 2, 8, ns, 256)
    f = _flags()
    m, l, a = run_dsa(c, num_splits=ns, chunk=ch, partials=True, flags=f)
    assert int(f.item()) & FP32_PATH
    # the maxima and sums within the per-head bound of the query rounding (the
    # tensor-core CTAs) or far inside it (the FP32 ones)
    bnd = lse_bound(c.q, c.k_scale, c.scale_kind, 2, c.sigma).reshape(4, 2, 8)
    bnd = np.repeat(bnd[:, :, None, :], ns, axis=2).reshape(8, ns, 8)
    assert np.all(np.abs(m - rm) <= bnd + 1e-6 * np.abs(rm))
    lr = l * np.exp(m - rm)
    assert np.all(np.abs(np.log(lr / rl)) <= bnd + 1e-5)
    # normalised partials, relative to the value scale of each channel
    on = a / l[..., None]
    rn = ra / rl[..., None]
    vsc = np.repeat(c.v_scale[None, :, None, None, :].astype(np.float64), 4, axis=0)
    vsc = np.broadcast_to(vsc.reshape(4, 2, 1, 1, 256), (4, 2, ns, 8, 256)).reshape(8, ns, 8, 256)
    assert np.max(np.abs(on - rn) / (127 * vsc)) < 2e-3


@pytest.mark.parametrize("kw", [dict(num_splits=1, chunk=512), dict(num_splits=4, chunk=128),
                                dict(prefill=True), dict(prefill=True, staged=True, num_splits=1),
                                dict(prefill=True, staged=True, num_splits=3)],
                         ids=["decode-1", "decode-4", "prefill", "prefill-staged",
                              "prefill-staged-3"])
def test_non_finite_value_scale_takes_the_fp32_path(K, kw):
    """One channel of KV head 1 has value scale +inf: that head's CTAs take
    the FP32 path (its output channel is not finite, as the FP64 result is
    not), and every other output and every lse still match the oracle."""
    c = W.random_sparse(seed=71, S=6, Hq=24, Hkv=2, D=256, N=900, max_sel=300, sink=True,
                        sigma=1.0 / 16)
    assert c.scale_kind == W.SCALE_PER_CHANNEL
    c.v_scale = c.v_scale.copy()
    c.v_scale[1, 5] = np.inf
    with np.errstate(invalid="ignore"):
        ref_o, ref_l = oracle_dsa(c)
    f = _flags()
    o, l = run_dsa(c, flags=f, **kw)
    assert int(f.item()) & FP32_PATH, kw
    bad = np.zeros(o.shape, bool)
    bad[:, 12:, 5] = True
    assert not np.isfinite(ref_o[bad]).any()
    assert not np.isfinite(o[bad]).any(), kw
    assert np.all(np.abs(o[~bad] - ref_o[~bad]) <= 2e-3 + 1e-2 * np.abs(ref_o[~bad])), kw
    assert_lse_close(l, ref_l, 1e-4)
