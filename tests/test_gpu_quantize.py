"""reshape_and_cache (quantize-on-write) on the GPU: bit-exact codes against
the oracle, and a decode over a cache written by it."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_close_oracle, dev, oracle_paged, run_paged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()
    return K


@pytest.mark.parametrize("kind", [W.SCALE_PER_TENSOR, W.SCALE_PER_CHANNEL])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_codes_bit_exact(K, kind, D):
    rng = np.random.default_rng(D + kind)
    nb, bs, Hkv, T = 40, 16, 4, 300
    kc = rng.integers(-127, 128, size=(nb, bs, Hkv, D)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(nb, bs, Hkv, D)).astype(np.int8)
    kn = (rng.standard_normal((T, Hkv, D)) * 2).astype(np.float16)
    vn = (rng.standard_normal((T, Hkv, D)) * 2).astype(np.float16)
    # exact ties at scale 0.5, saturation, non-finite values
    kn[0, 0, :8] = np.array([0.25, 0.75, -0.25, 1.25, 300, -300, np.nan, np.inf], np.float16)
    if kind == W.SCALE_PER_TENSOR:
        ks, vs = np.array([0.5], np.float32), np.array([0.0173], np.float32)
    else:
        ks = np.exp(rng.uniform(-5, 0, size=(Hkv, D))).astype(np.float32)
        ks[0, :8] = 0.5
        vs = np.exp(rng.uniform(-5, 0, size=(Hkv, D))).astype(np.float32)
    slots = rng.permutation(nb * bs)[:T].astype(np.int32)
    slots[5] = -1
    slots[9] = -3
    slots[11] = nb * bs + 2  # out of the pool
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd, vd = dev(kc), dev(vc)
    K.reshape_and_cache(dev(kn), dev(vn), dev(slots), kd, vd, dev(ks), dev(vs), kind, flags=flags)
    torch.cuda.synchronize()
    k_ref, v_ref = oracle.reshape_and_cache(kn, vn, slots, kc, vc, ks, vs, kind)
    np.testing.assert_array_equal(kd.cpu().numpy(), k_ref)
    np.testing.assert_array_equal(vd.cpu().numpy(), v_ref)
    assert int(flags.item()) & 0x8


def test_zero_tokens_is_a_no_op(K):
    z = torch.zeros((0, 2, 64), dtype=torch.float16, device="cuda")
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.int8, device="cuda")
    K.reshape_and_cache(z, z, torch.zeros(0, dtype=torch.int32, device="cuda"), kc, kc.clone(),
                        torch.ones(1, device="cuda"), torch.ones(1, device="cuda"), 1)
    assert int(kc.abs().sum()) == 0


def test_decode_over_a_cache_written_on_the_device(K):
    """Append one decode step's token per sequence with reshape_and_cache, then
    run paged_decode; compare with the oracle on the oracle-written cache."""
    c = W.random_paged(seed=21, B=4, Hq=16, Hkv=4, D=128, bs=16, max_blocks=32,
                       lens=[100, 257, 31, 500], sink=True, spare_blocks=6)
    rng = np.random.default_rng(3)
    kn = rng.standard_normal((4, 4, 128)).astype(np.float16)
    vn = rng.standard_normal((4, 4, 128)).astype(np.float16)
    # the new token of sequence b goes to position len_b
    slots = np.array([c.block_table[b, int(L) // 16] * 16 + int(L) % 16
                      for b, L in enumerate(c.seq_lens)], np.int32)
    assert np.all(c.block_table[np.arange(4), c.seq_lens // 16] >= 0)
    kd, vd = dev(c.k_cache), dev(c.v_cache)
    K.reshape_and_cache(dev(kn), dev(vn), dev(slots), kd, vd, dev(c.k_scale), dev(c.v_scale),
                        c.scale_kind)
    k_ref, v_ref = oracle.reshape_and_cache(kn, vn, slots, c.k_cache, c.v_cache, c.k_scale,
                                            c.v_scale, c.scale_kind)
    np.testing.assert_array_equal(kd.cpu().numpy(), k_ref)
    import dataclasses
    c2 = dataclasses.replace(c, k_cache=k_ref, v_cache=v_ref, seq_lens=c.seq_lens + 1)
    ref_o, _ = oracle_paged(c2)
    d = dict(q=dev(c2.q), k=kd, v=vd, ks=dev(c2.k_scale), vs=dev(c2.v_scale),
             bt=dev(c2.block_table), lens=dev(c2.seq_lens), sink=dev(c2.sink))
    o, _ = run_paged(c2, d, num_splits=0)
    assert_close_oracle(o, ref_o, "decode after quantize-on-write")
