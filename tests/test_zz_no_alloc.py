"""dsa_decode_static_workspace: the decode entry point for callers that cannot
allocate device memory at call time (for example an engine step that must not
allocate, or code with no access to the application's allocator).  It keeps
its split partials in a fixed device array inside the library instead of a
caller-supplied workspace.

The test calls it through the C ABI twice in a row, on two different
workloads (so the second call runs over the first call's leftovers in the
shared array), and compares each output with the ordinary dsa_decode on the
same inputs, within the tolerance of the other parity tests.  It also checks
that a geometry whose partials do not fit the fixed array is refused.
"""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import ATOL, RTOL, sparse_to_device

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
    out = torch.empty_like(d["q"])
    lse = torch.empty(S, Hq, dtype=torch.float32, device="cuda")
    K.dsa_decode_static_workspace(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind,
                                  d["idx"], c.sigma, d["sink"], num_splits=ns, chunk=chunk,
                                  out=out, lse=lse)
    return out, lse


def _close(a, b):
    a = a.float().cpu().numpy()
    b = b.float().cpu().numpy()
    assert np.all(np.isfinite(a))
    assert np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b))


def test_two_calls_in_a_row_match_the_ordinary_entry_point(K):
    cases = [
        # sparse decode, 8 rows, 24/2 heads, head_dim 256, 2048 candidates: 16 splits
        (W.sparse_decode(8, seed=3), 16, 128),
        # a different shape and geometry on the same array: 3 rows, 8/2 heads, D 128
        (W.random_sparse(seed=4, S=3, Hq=8, Hkv=2, D=128, N=900, max_sel=700,
                         invalid_frac=0.1, sink=True), 11, 64),
    ]
    for c, ns, chunk in cases:
        d = sparse_to_device(c)
        want, want_lse = _ordinary(K, c, d, ns, chunk)
        got, got_lse = _static(K, c, d, ns, chunk)
        torch.cuda.synchronize()
        _close(got, want)
        g, w = got_lse.cpu().numpy(), want_lse.cpu().numpy()
        assert np.all(np.abs(g - w) <= 1e-4 * np.maximum(1.0, np.abs(w)))


def test_automatic_geometry(K):
    c = W.sparse_decode(2, seed=5)
    d = sparse_to_device(c)
    ns, chunk, _, _ = K.decode_plan(K.PATH_DSA, K.CACHE_INT8, c.idx.shape[1], 2, 24, 2, 256,
                                    K.GEOM_POW2_TILES)
    want, _ = _ordinary(K, c, d, ns, chunk)
    got, _ = _static(K, c, d, 0, 0)
    torch.cuda.synchronize()
    _close(got, want)


def test_geometry_beyond_the_fixed_size_is_refused(K):
    c = W.random_sparse(seed=6, S=16, Hq=24, Hkv=2, D=256, N=4000, max_sel=2048)
    need = K.split_workspace_bytes(16 * 2, 32, 12, 256)
    assert need > K.STATIC_WORKSPACE_BYTES
    d = sparse_to_device(c)
    with pytest.raises(K.Int8KVError) as e:
        _static(K, c, d, 32, 64)
    assert e.value.status == 4  # I8KV_EWORKSPACE, nothing enqueued
