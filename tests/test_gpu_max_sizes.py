"""Caches larger than 2^32 bytes: the gathers address rows whose byte offsets
need 64 bits.

The caches are filled on the device; the oracle sees only the rows the lists
or tables reference (copied back and re-indexed into a small case of the same
attention), so its result is the attention over exactly those rows.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_close_oracle, dev, oracle_dsa, oracle_paged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()
    return K


def _free_gb():
    free, _ = torch.cuda.mem_get_info()
    return free / 2 ** 30


def test_sparse_decode_rows_beyond_4_gib(K):
    if _free_gb() < 12:
        pytest.skip("needs 12 GiB of free device memory")
    N, Hkv, D, Hq, S, n = 9_000_000, 2, 256, 8, 3, 300   # 4.6 GB per cache tensor
    g = torch.Generator(device="cuda").manual_seed(0)
    kc = torch.randint(-127, 128, (N, Hkv, D), dtype=torch.int8, device="cuda", generator=g)
    vc = torch.randint(-127, 128, (N, Hkv, D), dtype=torch.int8, device="cuda", generator=g)
    rng = np.random.default_rng(1)
    # lists reaching the last rows (byte offsets above 2^32) and some low rows
    rows = np.concatenate([N - 1 - rng.choice(200_000, size=(S, n - 20), replace=False),
                           rng.choice(1000, size=(S, 20), replace=False)], axis=1).astype(np.int32)
    ks = np.exp(rng.uniform(-5, -3, size=(Hkv, D))).astype(np.float32)
    vs = np.exp(rng.uniform(-5, -3, size=(Hkv, D))).astype(np.float32)
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    out = torch.empty((S, Hq, D), dtype=torch.float16, device="cuda")
    lse = torch.empty((S, Hq), dtype=torch.float32, device="cuda")
    ns, ch, wsb, _ = K.decode_plan(K.PATH_DSA, K.CACHE_INT8, n, S, Hq, Hkv, D,
                                   K.GEOM_POW2_TILES)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    K.dsa_decode(dev(q), kc, vc, dev(ks), dev(vs), W.SCALE_PER_CHANNEL, dev(rows), 1 / 16,
                 num_splits=ns, chunk=ch, workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    # the referenced rows, re-indexed 0 .. U-1
    uniq, inv = np.unique(rows, return_inverse=True)
    sel = torch.from_numpy(uniq.astype(np.int64)).cuda()
    small = W.SparseCase(q=q, k_codes=kc[sel].cpu().numpy(), v_codes=vc[sel].cpu().numpy(),
                         k_scale=ks, v_scale=vs, scale_kind=W.SCALE_PER_CHANNEL,
                         idx=inv.reshape(rows.shape).astype(np.int32), sigma=1 / 16, sink=None)
    ref_o, _ = oracle_dsa(small)
    assert_close_oracle(out.float().cpu().numpy().astype(np.float64), ref_o, "rows beyond 4 GiB")


def test_paged_decode_blocks_beyond_4_gib(K):
    if _free_gb() < 12:
        pytest.skip("needs 12 GiB of free device memory")
    nb, bs, Hkv, D, Hq, B, mb = 2 ** 21 + 64, 16, 1, 128, 8, 3, 40   # 4.3 GB per cache tensor
    g = torch.Generator(device="cuda").manual_seed(2)
    kc = torch.randint(-127, 128, (nb, bs, Hkv, D), dtype=torch.int8, device="cuda", generator=g)
    vc = torch.randint(-127, 128, (nb, bs, Hkv, D), dtype=torch.int8, device="cuda", generator=g)
    rng = np.random.default_rng(3)
    lens = np.array([640, 333, 17], np.int32)
    bt = np.full((B, mb), -1, np.int32)
    for b in range(B):
        nblk = -(-int(lens[b]) // bs)
        bt[b, :nblk] = nb - 1 - rng.choice(5000, size=nblk, replace=False)  # top blocks
    ks = np.exp(rng.uniform(-5, -3, size=(Hkv, D))).astype(np.float32)
    vs = np.exp(rng.uniform(-5, -3, size=(Hkv, D))).astype(np.float32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    sink = rng.standard_normal(Hq).astype(np.float32)
    out = torch.empty((B, Hq, D), dtype=torch.float16, device="cuda")
    ns, ch, wsb, _ = K.decode_plan(K.PATH_PAGED, K.CACHE_INT8, mb * bs, B, Hq, Hkv, D,
                                   K.GEOM_WAVE)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    K.paged_decode(dev(q), kc, vc, dev(ks), dev(vs), W.SCALE_PER_CHANNEL, dev(bt), dev(lens),
                   1 / np.sqrt(D), dev(sink), num_splits=ns, chunk=ch, workspace=ws, out=out)
    torch.cuda.synchronize()
    used = np.unique(bt[bt >= 0])
    sel = torch.from_numpy(used.astype(np.int64)).cuda()
    remap = {int(b): i for i, b in enumerate(used)}
    small_bt = np.vectorize(lambda b: remap.get(int(b), -1))(bt).astype(np.int32)
    small = W.PagedCase(q=q, k_cache=kc[sel].cpu().numpy(), v_cache=vc[sel].cpu().numpy(),
                        k_scale=ks, v_scale=vs, scale_kind=W.SCALE_PER_CHANNEL,
                        block_table=small_bt, seq_lens=lens, sigma=1 / float(np.sqrt(D)),
                        sink=sink)
    ref_o, _ = oracle_paged(small)
    assert_close_oracle(out.float().cpu().numpy().astype(np.float64), ref_o, "blocks beyond 4 GiB")


def test_quantize_on_write_slots_beyond_4_gib(K):
    if _free_gb() < 10:
        pytest.skip("needs 10 GiB of free device memory")
    num_slots, Hkv, D, T = 2 ** 25 + 8, 1, 128, 64     # 4.3 GB per cache tensor
    kc = torch.zeros((num_slots, Hkv, D), dtype=torch.int8, device="cuda")
    vc = torch.zeros((num_slots, Hkv, D), dtype=torch.int8, device="cuda")
    rng = np.random.default_rng(4)
    kn = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    vn = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    slots = (num_slots - 1 - rng.choice(1000, size=T, replace=False)).astype(np.int32)
    ks = np.array([0.02], np.float32)
    vs = np.array([0.03], np.float32)
    K.reshape_and_cache(dev(kn), dev(vn), dev(slots), kc, vc, dev(ks), dev(vs),
                        W.SCALE_PER_TENSOR)
    torch.cuda.synchronize()
    sel = torch.from_numpy(slots.astype(np.int64)).cuda()
    z = np.zeros((T, Hkv, D), np.int8)
    k_ref, v_ref = oracle.reshape_and_cache(kn, vn, np.arange(T, dtype=np.int32), z, z, ks, vs,
                                            W.SCALE_PER_TENSOR)
    np.testing.assert_array_equal(kc[sel].cpu().numpy(), k_ref)
    np.testing.assert_array_equal(vc[sel].cpu().numpy(), v_ref)
    # nothing else was written near them
    assert int(kc[num_slots - 1001:].ne(0).any(dim=(1, 2)).sum()) == T
