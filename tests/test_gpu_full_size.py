"""Parity at the full sizes of the benchmark workloads, in the launch
configuration the benchmark times (the automatic geometry of the library).

* sparse-candidate decode, S = 1, 2, 4, 8 rows, 24/2 heads, D 256, a
  16384-token cache and 2048 candidates per row: every output;
* paged INT8 (and float8 e4m3fn) decode of 16 sequences with lengths
  U[512, 8192]: every output;
* deep context, 16 rows, live 2600 of cap 4096, int8 / e4m3fn / fp16 cache,
  adaptive and fixed chunks: every output, and each split count against the
  single split;
* sparse prefill, 2048 rows over an 8192-token cache: the GPU runs all rows,
  the oracle checks 64 of them, one by one; and the other row counts and
  contexts the benchmark times (128 / 8192 rows, 8192 / 32768 positions),
  each on the path and split count the library picks, on sampled rows.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_close_oracle, assert_lse_close, assert_lse_oracle, assert_split_close,
                     lse_bound, oracle_dsa, oracle_paged, paged_bound, paged_to_device, run_dsa,
                     run_paged, sparse_to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()


def _sparse_bound(c):
    return lse_bound(c.q, c.k_scale, c.scale_kind, c.k_codes.shape[1], c.sigma)


@pytest.mark.parametrize("S", [1, 2, 4, 8])
def test_sparse_decode_full_size(S):
    c = W.sparse_decode(S, seed=0)
    ref_o, ref_l = oracle_dsa(c)
    d = sparse_to_device(c)
    o, l = run_dsa(c, d)  # automatic geometry (power-of-two tiles), as timed
    assert_close_oracle(o, ref_o, f"S {S}")
    assert_lse_oracle(l, ref_l, _sparse_bound(c))
    o1, l1 = run_dsa(c, d, num_splits=1, chunk=2048)
    assert_split_close(o, o1, f"S {S} auto vs one split")
    assert_lse_close(l, l1, 1e-4)


@pytest.mark.parametrize("cache", ["int8", "fp8"])
def test_paged_decode_full_size(cache):
    c = W.paged_decode(seed=0, cache=cache)
    ref_o, ref_l = oracle_paged(c)
    d = paged_to_device(c)
    o, l = run_paged(c, d)  # automatic geometry (wave rule), as timed
    assert_close_oracle(o, ref_o, f"paged {cache}")
    assert_lse_oracle(l, ref_l, paged_bound(c))
    o1, l1 = run_paged(c, d, num_splits=1, chunk=8192)
    assert_split_close(o, o1, f"paged {cache} auto vs one split")
    assert_lse_close(l, l1, 1e-4)


@pytest.mark.parametrize("cache", ["int8", "fp8", "fp16"])
def test_deep_context_full_size(cache):
    import int8_kv_cache_gb300 as K
    c = W.deep_context(seed=0, cache=cache)
    ref_o, ref_l = oracle_paged(c)
    d = paged_to_device(c)
    o1, l1 = run_paged(c, d, num_splits=1, chunk=4096)
    assert_close_oracle(o1, ref_o, f"deep {cache} one split")
    for ovr in (0, 128, 256, 512):
        dt = {"int8": K.CACHE_INT8, "fp8": K.CACHE_FP8, "fp16": K.CACHE_FP16}[cache]
        ns, ch, _, _ = K.decode_plan(K.PATH_PAGED, dt, 4096, 16, 16, 2, 128, K.GEOM_WAVE, ovr)
        o, l = run_paged(c, d, num_splits=ns, chunk=ch)
        assert_close_oracle(o, ref_o, f"deep {cache} chunk {ch}")
        assert_lse_oracle(l, ref_l, paged_bound(c))
        assert_split_close(o, o1, f"deep {cache} chunk {ch} vs one split")
        assert_lse_close(l, l1, 1e-4)


@pytest.mark.parametrize("staged", [False, True], ids=["converting", "staged"])
def test_sparse_prefill_full_size_sampled_rows(staged):
    c = W.sparse_prefill(seed=0)
    o, l = run_dsa(c, prefill=True, staged=staged)
    rows = np.linspace(0, c.q.shape[0] - 1, 64).astype(np.int64)
    sub = dataclasses.replace(c, q=c.q[rows], idx=c.idx[rows])
    ref_o, ref_l = oracle_dsa(sub)
    assert_close_oracle(o[rows], ref_o, "prefill sampled rows")
    assert_lse_oracle(l[rows], ref_l, _sparse_bound(sub))


@pytest.mark.parametrize("rows,N,literal", [(128, 8192, False), (8192, 8192, False),
                                            (128, 32768, False), (2048, 32768, False),
                                            (8192, 32768, False), (2048, 8192, True)])
def test_sparse_prefill_table_sampled_rows(rows, N, literal):
    # the library's own choice for each shape: the tensor-core kernel (split 6
    # ways at 128 rows) where the lists cover a quarter of the cache, else the
    # gathering kernel; and the literal reading (row i at position i)
    c = W.sparse_prefill(seed=0, rows=rows, N=N, literal=literal)
    o, l = run_dsa(c, prefill=True, staged=True)
    sample = np.linspace(0, rows - 1, 16).astype(np.int64)
    sub = dataclasses.replace(c, q=c.q[sample], idx=c.idx[sample])
    ref_o, ref_l = oracle_dsa(sub)
    assert_close_oracle(o[sample], ref_o, f"prefill {rows} x {N}")
    assert_lse_oracle(l[sample], ref_l, _sparse_bound(sub))
