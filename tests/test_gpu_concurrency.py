"""Calls from two host threads on two streams at once (the library is
re-entrant: its only shared state is a per-device attribute cache behind a
mutex), each with its own workspace: results bit-identical to serial calls."""
import threading

import numpy as np
import pytest
import torch

import workloads as W
from helpers import paged_to_device, sparse_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()
    return K


def test_two_threads_two_streams_match_serial_calls(K):
    cs = W.sparse_decode(4, seed=7)
    cp = W.random_paged(seed=8, B=6, Hq=16, Hkv=2, D=128, bs=16, max_blocks=64,
                        lens=[1000, 3, 512, 777, 0, 1024], sink=True)
    ds, dp = sparse_to_device(cs), paged_to_device(cp)
    ns_s, ch_s, wsb_s, _ = K.decode_plan(K.PATH_DSA, K.CACHE_INT8, 2048, 4, 24, 2, 256,
                                         K.GEOM_POW2_TILES)
    ns_p, ch_p, wsb_p, _ = K.decode_plan(K.PATH_PAGED, K.CACHE_INT8, 1024, 6, 16, 2, 128,
                                         K.GEOM_WAVE)

    def sparse(stream, ws, out):
        with torch.cuda.stream(stream):
            for _ in range(50):
                K.dsa_decode(ds["q"], ds["k"], ds["v"], ds["ks"], ds["vs"], cs.scale_kind,
                             ds["idx"], cs.sigma, num_splits=ns_s, chunk=ch_s, workspace=ws,
                             out=out, stream=stream)

    def paged(stream, ws, out):
        with torch.cuda.stream(stream):
            for _ in range(50):
                K.paged_decode(dp["q"], dp["k"], dp["v"], dp["ks"], dp["vs"], cp.scale_kind,
                               dp["bt"], dp["lens"], cp.sigma, dp["sink"], num_splits=ns_p,
                               chunk=ch_p, workspace=ws, out=out, stream=stream)

    def bufs():
        return (torch.empty(wsb_s // 4, dtype=torch.float32, device="cuda"),
                torch.empty_like(ds["q"]),
                torch.empty(wsb_p // 4, dtype=torch.float32, device="cuda"),
                torch.empty_like(dp["q"]))

    s0 = torch.cuda.current_stream()
    a = bufs()
    sparse(s0, a[0], a[1])
    paged(s0, a[2], a[3])
    torch.cuda.synchronize()

    b = bufs()
    st1, st2 = torch.cuda.Stream(), torch.cuda.Stream()
    errors = []

    def run(fn, *args):
        try:
            fn(*args)
        except Exception as e:  # surfaced below
            errors.append(e)
    t1 = threading.Thread(target=run, args=(sparse, st1, b[0], b[1]))
    t2 = threading.Thread(target=run, args=(paged, st2, b[2], b[3]))
    t1.start()
    t2.start()
    t1.join()
    t2.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert torch.equal(a[1], b[1])
    assert torch.equal(a[3], b[3])
