"""dsa_decode_static_workspace: the decode entry point for callers that cannot
allocate device memory at call time (for example an engine step that must not
allocate, or code with no access to the application's allocator).  It keeps
its split partials in a fixed device array inside the library instead of a
caller-supplied workspace.

The static calls run the same kernels under the same geometry as the ordinary
dsa_decode, so their outputs must be identical bit for bit.  The first test
queues two static calls back to back on one stream, with no synchronisation in
between (the second call's decode kernel follows the first call's combine
kernel over the one shared array), then compares both outputs with ordinary
calls on the same inputs.  A partial left over from one call and read by the
next would show up as a difference.  The other tests check the automatic
geometry, that a geometry whose partials do not fit the array is refused, and
that a call with no output pointer is refused before anything is enqueued.
"""
import ctypes

import pytest
import torch

import workloads as W
from helpers import sparse_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()
    return K


def _ordinary(K, c, d, ns, chunk):
    S, Hq, D = c.q.shape
    Hkv = c.k_codes.shape[1]
    wsb = K.split_workspace_bytes(S * Hkv, ns, Hq // Hkv, D)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    out = torch.empty_like(d["q"])
    lse = torch.empty(S, Hq, dtype=torch.float32, device="cuda")
    K.dsa_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                 d["sink"], num_splits=ns, chunk=chunk, workspace=ws, out=out, lse=lse)
    return out, lse


def _static(K, c, d, ns, chunk):
    S, Hq, _ = c.q.shape
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device="cuda")
    K.dsa_decode_static_workspace(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind,
                                  d["idx"], c.sigma, d["sink"], num_splits=ns, chunk=chunk,
                                  out=out, lse=lse)
    return out, lse


def _identical(got, want):
    (o, l), (wo, wl) = got, want
    assert torch.equal(o, wo), "output differs from the ordinary entry point"
    assert torch.equal(l, wl), "lse differs from the ordinary entry point"


def test_two_calls_back_to_back_match_the_ordinary_entry_point(K):
    cases = [
        # sparse decode, 8 rows, 24/2 heads, head_dim 256, 2048 candidates: 16 splits
        (W.sparse_decode(8, seed=3), 16, 128),
        # a different shape and geometry over the same array: 3 rows, 8/2 heads, D 128
        (W.random_sparse(seed=4, S=3, Hq=8, Hkv=2, D=128, N=900, max_sel=700,
                         invalid_frac=0.1, sink=True), 11, 64),
        # the first shape again with other inputs: the array still holds the
        # first call's partials of this geometry
        (W.sparse_decode(8, seed=5), 16, 128),
    ]
    devs = [sparse_to_device(c) for c, _, _ in cases]
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        # all static calls queued on one stream, nothing waited on in between
        got = [_static(K, c, d, ns, ch) for (c, ns, ch), d in zip(cases, devs)]
        want = [_ordinary(K, c, d, ns, ch) for (c, ns, ch), d in zip(cases, devs)]
    stream.synchronize()
    for g, w in zip(got, want):
        _identical(g, w)


def test_automatic_geometry(K):
    c = W.sparse_decode(2, seed=5)
    d = sparse_to_device(c)
    ns, chunk, _, _ = K.decode_plan(K.PATH_DSA, K.CACHE_INT8, c.idx.shape[1], 2, 24, 2, 256,
                                    K.GEOM_POW2_TILES)
    assert ns > 1
    want = _ordinary(K, c, d, ns, chunk)
    got = _static(K, c, d, 0, 0)
    torch.cuda.synchronize()
    _identical(got, want)


def test_geometry_beyond_the_fixed_size_is_refused(K):
    c = W.random_sparse(seed=6, S=16, Hq=24, Hkv=2, D=256, N=4000, max_sel=2048)
    need = K.split_workspace_bytes(16 * 2, 32, 12, 256)
    assert need > K.STATIC_WORKSPACE_BYTES
    d = sparse_to_device(c)
    with pytest.raises(K.Int8KVError) as e:
        _static(K, c, d, 32, 64)
    assert e.value.status == 4  # I8KV_EWORKSPACE, nothing enqueued


def test_missing_output_is_refused(K):
    # through the C ABI directly: out = NULL with rows to decode would leave the
    # partials in the library's private array, so the call refuses it
    c = W.sparse_decode(1, seed=7)
    d = sparse_to_device(c)
    S, Hq, D = c.q.shape
    N, Hkv, _ = c.k_codes.shape
    st = K.load().dsa_decode_static_workspace(
        d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["ks"].data_ptr(),
        d["vs"].data_ptr(), c.scale_kind, d["idx"].data_ptr(), S, Hq, Hkv, D, N,
        c.idx.shape[1], ctypes.c_float(c.sigma), None, 4, 512, None, None, None,
        torch.cuda.current_stream().cuda_stream)
    assert st == 1  # I8KV_EINVAL
