"""The dense tensor-core prefill (dsa_prefill for head_dim 128 / 256 when the
rows' lists cover the cache densely enough) against the FP64 oracle, on the
cases its design has to get right: unsorted lists with invalid entries, lists
that repeat an entry (those rows go to the FP32 path), empty rows, a last tile
only partly filled with query vectors, one query head per KV head (tiles that
span 128 rows), per-tensor scales, the head sink, and a large value scale with
a deep candidate.  The full-size workload is covered by test_gpu_full_size."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import (assert_close_oracle, assert_lse_close, assert_lse_oracle, assert_split_close,
                     lse_bound, oracle_dsa, run_dsa)

pytestmark = pytest.mark.gpu

FP32_PATH = 0x10
WAIT_TIMEOUT = 0x20


def bound_of(c):
    """lse tolerance against the oracle: the query-rounding bound per head."""
    return lse_bound(c.q, c.k_scale, c.scale_kind, c.k_codes.shape[1], c.sigma)


def _flags():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _run(c, form=(False, 0)):
    """form: (staged, num_splits); the converting form is unsplit."""
    f = _flags()
    o, l = run_dsa(c, prefill=True, flags=f, staged=form[0], num_splits=form[1])
    return o, l, int(f.item())


# both forms of the kernel: converting the int8 cache in every CTA, and staged
# (fp16 operand images made once per call in a workspace), the latter with the
# automatic split count (small cases: up to 8 splits per tile), unsplit, and
# with 5 splits
@pytest.fixture(params=[(False, 0), (True, 0), (True, 1), (True, 5)],
                ids=["converting", "staged", "staged-unsplit", "staged-5"])
def staged(request):
    return request.param


@pytest.mark.parametrize("S,Hq,Hkv,D,N,max_sel,kind", [
    (37, 24, 2, 256, 700, 400, W.SCALE_PER_CHANNEL),   # 444 vectors per KV head: partial tile
    (20, 8, 2, 128, 1000, 300, W.SCALE_PER_TENSOR),
    (3, 2, 2, 256, 500, 200, W.SCALE_PER_CHANNEL),     # G = 1: a tile spans 128 rows
    (130, 1, 1, 128, 256, 64, W.SCALE_PER_CHANNEL),    # G = 1, two tiles
])
def test_unsorted_lists_with_invalid_entries(S, Hq, Hkv, D, N, max_sel, kind, staged):
    c = W.random_sparse(seed=S * 7 + D, S=S, Hq=Hq, Hkv=Hkv, D=D, N=N, max_sel=max_sel,
                        invalid_frac=0.15, scale_kind=kind, sink=True, sigma=1.0 / 16)
    ref_o, ref_l = oracle_dsa(c)
    o, l, f = _run(c, staged)
    assert not f & WAIT_TIMEOUT
    assert_close_oracle(o, ref_o, "dense prefill")
    assert_lse_oracle(l, ref_l, bound_of(c))


def test_repeated_entries_and_empty_rows(staged):
    c = W.random_sparse(seed=11, S=24, Hq=24, Hkv=2, D=256, N=600, max_sel=256, sink=True,
                        sigma=1.0 / 16)
    c.idx[3, 10:20] = c.idx[3, 0:10]        # row 3 lists ten candidates twice
    c.idx[7, 100] = c.idx[7, 5]             # row 7 one candidate twice
    c.idx[12, :] = -1                       # row 12 attends nothing
    c.idx[13, :] = 600 + np.arange(256)     # row 13: every entry out of range
    ref_o, ref_l = oracle_dsa(c)
    o, l, f = _run(c, staged)
    assert f & FP32_PATH                     # the repeating rows took the FP32 path
    assert not f & WAIT_TIMEOUT
    assert_close_oracle(o, ref_o, "repeated entries")
    assert np.all(o[12] == 0) and np.all(np.isneginf(l[12]))
    assert np.all(o[13] == 0) and np.all(np.isneginf(l[13]))
    assert_lse_close(l, ref_l, 1e-4)


def test_matches_the_decode_kernel_on_the_same_rows():
    # the prefill's dense kernel and the decode kernel (one split) compute the
    # same quantity with different tensor-core paths
    c = W.random_sparse(seed=12, S=40, Hq=24, Hkv=2, D=256, N=1024, max_sel=512,
                        sorted_lists=True, sigma=1.0 / 16)
    o, l, _ = _run(c)
    od, ld = run_dsa(c, num_splits=1, chunk=512)
    assert np.all(np.abs(o - od) <= 2e-3 + 1e-2 * np.abs(od))
    assert_lse_close(l, ld, 1e-4)


@pytest.mark.parametrize("q0,vs,fp32", [(336.0, 2.0 ** 28, True), (320.0, 2.0 ** 28, False)])
def test_tail_depth_rule(q0, vs, fp32, staged):
    """A candidate 21 nats below the maximum under a value scale of 2^28 goes to
    the FP32 path; exactly 20 nats down stays on the tensor cores.  (Split, the
    rule holds per split, against the split's own running maximum: where the
    two candidates fall in different splits, each is its split's maximum and
    the merge weighs them in FP32, so no split needs the FP32 path.)"""
    c = W.tiny_probability_case(q0, 1, vs, D=128)
    c.q = np.concatenate([c.q] * 2, axis=1)  # 8 query heads over 2 KV heads
    c.k_codes = np.concatenate([c.k_codes] * 2, axis=1)
    c.v_codes = np.concatenate([c.v_codes] * 2, axis=1)
    ref_o, ref_l = oracle_dsa(c)
    o, l, f = _run(c, staged)
    if not staged[0] or staged[1] == 1:
        assert bool(f & FP32_PATH) == fp32
    assert np.all(np.abs(o - ref_o) <= 2e-3 + 1e-2 * np.abs(ref_o))
    assert_lse_close(l, ref_l, 1e-5)


@pytest.mark.parametrize("S,Hq,Hkv,D,N,max_sel", [
    (50, 16, 1, 128, 333, 120),    # G = 16: a tile spans 9 rows; N not a multiple of 128
    (9, 12, 1, 256, 129, 40),      # one selected position in the last, 1-token block
    (4, 8, 2, 256, 2000, 300),     # 4 * max_sel < N: the gathering kernel serves it
    (6, 8, 2, 64, 200, 100),       # head_dim 64: the gathering kernel serves it
])
def test_shapes_on_either_kernel(S, Hq, Hkv, D, N, max_sel, staged):
    c = W.random_sparse(seed=S + N, S=S, Hq=Hq, Hkv=Hkv, D=D, N=N, max_sel=max_sel,
                        invalid_frac=0.05, sink=True, sigma=1.0 / 16)
    if N == 129:
        c.idx[0, 0] = 128  # the only position of the last block
    ref_o, ref_l = oracle_dsa(c)
    o, l, f = _run(c, staged)
    assert not f & WAIT_TIMEOUT
    assert_close_oracle(o, ref_o, "prefill shape")
    assert_lse_oracle(l, ref_l, bound_of(c))


def test_prefill_can_be_captured_and_replayed():
    # the kernel choice and its launch depend on shapes only: a captured call
    # replays to the same result as an eager one, over new inputs
    import int8_kv_cache_gb300 as K
    from helpers import sparse_to_device
    c = W.random_sparse(seed=21, S=30, Hq=24, Hkv=2, D=256, N=700, max_sel=300, sigma=1.0 / 16)
    d = sparse_to_device(c)
    out = torch.empty_like(d["q"])
    s = torch.cuda.Stream()

    def call():
        K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                      out=out)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    out.zero_()
    d["q"].copy_(torch.flip(d["q"], dims=[0]))  # new query rows, same buffer
    g.replay()
    torch.cuda.synchronize()
    flipped = out.clone()
    d["q"].copy_(torch.flip(d["q"], dims=[0]))  # back to the original rows
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert not torch.equal(flipped, eager)


@pytest.mark.parametrize("S,Hq,Hkv,D,N,max_sel", [
    (37, 24, 2, 256, 700, 400), (20, 8, 2, 128, 1000, 300), (130, 1, 1, 128, 256, 64),
])
def test_staged_form_is_bit_identical(S, Hq, Hkv, D, N, max_sel):
    # the operand images hold exactly what the converters write, and the
    # products and the softmax are the same code: the outputs agree bit for bit
    c = W.random_sparse(seed=S + 3, S=S, Hq=Hq, Hkv=Hkv, D=D, N=N, max_sel=max_sel,
                        invalid_frac=0.1, sink=True, sigma=1.0 / 16)
    o1, l1, f1 = _run(c, (False, 0))
    o2, l2, f2 = _run(c, (True, 1))
    assert f1 == f2
    assert np.array_equal(o1, o2, equal_nan=True)
    assert np.array_equal(l1, l2, equal_nan=True)


def test_staged_workspace_is_sized_and_checked():
    import ctypes
    import int8_kv_cache_gb300 as K
    from helpers import sparse_to_device
    c = W.random_sparse(seed=8, S=16, Hq=24, Hkv=2, D=256, N=300, max_sel=100, sigma=1.0 / 16)
    # Hkv x blocks x (K, V) x 128 x D x fp16, then the rows' bitmasks (16
    # bytes per block) and repeat flags
    stage = 2 * 3 * 2 * 128 * 256 * 2 + 16 * 3 * 16 + 16 * 4
    need = K.prefill_workspace_bytes(16, 24, 2, 256, 300, 100, 1)
    assert need == stage
    # automatic: 2 KV heads x 2 tiles of 128 vectors leave most SMs idle, so
    # each tile's blocks split min(8, SMs / 4) ways, with their partials
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ns = min(8, sms // 4)
    assert K.prefill_workspace_bytes(16, 24, 2, 256, 300, 100) == \
        (stage + 255) // 256 * 256 + 16 * 24 * ns * 258 * 4
    # enough tiles to fill the SMs: no split
    assert K.prefill_workspace_bytes(2048, 24, 2, 256, 8192, 2048) == \
        2 * 64 * 2 * 128 * 256 * 2 + 2048 * 64 * 16 + 2048 * 4
    d = sparse_to_device(c)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(K.Int8KVError, match="workspace"):
        K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                      workspace=ws[: need - 16], num_splits=1)
    with pytest.raises(K.Int8KVError, match="workspace"):
        K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                      workspace=ws, num_splits=2)  # no room for the partials
    with pytest.raises(K.Int8KVError):
        K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                      workspace=ws[8:], num_splits=1)  # not 16-byte aligned
    # the gathering kernel's shapes need none (and ignore one)
    assert K.prefill_workspace_bytes(16, 24, 2, 256, 3000, 100) == 0
    assert K.prefill_workspace_bytes(16, 8, 2, 64, 300, 100) == 0


def test_largest_cache_the_masks_allow(staged):
    # 16384 cache positions: 512 mask words per row and 128 blocks per tile,
    # near the shared-memory limit of the row masks at 12 query heads per KV
    # head (about 20k positions; longer caches take the gathering kernel)
    import int8_kv_cache_gb300 as K
    assert K.prefill_workspace_bytes(16, 24, 2, 256, 16384, 4096) > 0
    c = W.random_sparse(seed=31, S=16, Hq=24, Hkv=2, D=256, N=16384, max_sel=4096,
                        sigma=1.0 / 16)
    ref_o, ref_l = oracle_dsa(c)
    o, l, f = _run(c, staged)
    assert not f & WAIT_TIMEOUT
    assert_close_oracle(o, ref_o, "large cache")
    assert_lse_oracle(l, ref_l, bound_of(c))


@pytest.mark.parametrize("S,Hq,Hkv,D,N,max_sel", [
    (37, 24, 2, 256, 700, 400),    # partial last tile, 6 blocks
    (3, 2, 2, 256, 500, 200),      # G = 1
    (50, 16, 1, 128, 333, 120),    # N not a multiple of 128
    (9, 12, 1, 256, 256, 64),      # 2 blocks: most splits get none
])
def test_splits_agree_with_the_unsplit_kernel(S, Hq, Hkv, D, N, max_sel):
    # any split of a tile's blocks merges to the unsplit result (split vs
    # unsplit within 1e-3), and both match the oracle
    c = W.random_sparse(seed=S * 3 + N, S=S, Hq=Hq, Hkv=Hkv, D=D, N=N, max_sel=max_sel,
                        invalid_frac=0.1, sink=True, sigma=1.0 / 16)
    ref_o, ref_l = oracle_dsa(c)
    o1, l1, f1 = _run(c, (True, 1))
    assert not f1 & WAIT_TIMEOUT
    for ns in (2, 3, 8, 32):
        o, l, f = _run(c, (True, ns))
        assert not f & WAIT_TIMEOUT
        assert_close_oracle(o, ref_o, f"{ns} splits")
        assert_lse_oracle(l, ref_l, bound_of(c))
        assert_split_close(o, o1, f"{ns} splits vs one")
        assert_lse_close(l, l1, 1e-4)


def test_split_fp32_vectors_publish_partials():
    # rows that repeat entries, and every vector of a few rows over the
    # query-folding budget, go to the FP32 path in each split over that
    # split's positions; the merge matches the oracle
    c = W.random_sparse(seed=77, S=12, Hq=24, Hkv=2, D=256, N=900, max_sel=300,
                        invalid_frac=0.05, sink=True, sigma=1.0 / 16)
    c.idx[2, 20:30] = c.idx[2, 0:10]                           # repeated entries
    c.q[5] = (c.q[5].astype(np.float32) * 32).astype(np.float16)  # over the budget
    ref_o, ref_l = oracle_dsa(c)
    for ns in (1, 4, 7):
        o, l, f = _run(c, (True, ns))
        assert f & FP32_PATH and not f & WAIT_TIMEOUT
        assert_close_oracle(o, ref_o, f"{ns} splits")
        assert_lse_close(l, ref_l, 1e-4)


def test_split_prefill_can_be_captured_and_replayed():
    import int8_kv_cache_gb300 as K
    from helpers import sparse_to_device
    c = W.random_sparse(seed=22, S=10, Hq=24, Hkv=2, D=256, N=700, max_sel=300, sigma=1.0 / 16)
    d = sparse_to_device(c)
    out = torch.empty_like(d["q"])
    ws = torch.empty(K.prefill_workspace_bytes(10, 24, 2, 256, 700, 300), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()

    def call():
        K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                      out=out, workspace=ws)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    ref_o, _ = oracle_dsa(c)
    assert_close_oracle(out.float().cpu().numpy().astype(np.float64), ref_o, "captured splits")


@pytest.mark.parametrize("form", [(False, 0), (True, 1), (True, 4)],
                         ids=["converting", "staged-unsplit", "staged-4"])
def test_tiles_whose_rows_attend_nothing(form):
    # every list entry invalid in the first 20 rows (whole tiles of both KV
    # heads with no selected block) and in row 31: O = 0, lse = -inf there,
    # the other rows as the oracle
    c = W.random_sparse(seed=41, S=40, Hq=24, Hkv=2, D=256, N=600, max_sel=256, sink=True,
                        sigma=1.0 / 16)
    c.idx[:20] = -1
    c.idx[31] = 600 + np.arange(256)
    ref_o, ref_l = oracle_dsa(c)
    o, l, f = _run(c, form)
    assert not f & WAIT_TIMEOUT
    dead = np.zeros(40, bool)
    dead[:20] = True
    dead[31] = True
    assert np.all(o[dead] == 0) and np.all(np.isneginf(l[dead]))
    assert_close_oracle(o[~dead], ref_o[~dead], "live rows")
    assert_lse_close(l[~dead], ref_l[~dead], 1e-4)


@pytest.mark.parametrize("S,Hq,Hkv,D,N,max_sel,ns", [
    (37, 24, 2, 256, 700, 400, 3),   # tiles straddle rows; a partial last tile
    (3, 2, 2, 256, 500, 200, 4),     # G = 1: one tile spans every row
    (20, 8, 2, 128, 1000, 300, 5),
    (9, 12, 1, 256, 256, 64, 8),     # two blocks: most splits get none
])
def test_split_partials_match_the_oracle(S, Hq, Hkv, D, N, max_sel, ns):
    # each split CTA's published partial (the workspace after the images and
    # the row masks, in the decode's partial layout) against the oracle's
    # partial over the same position range: same emptiness, lse per split
    # within the query-rounding bound, normalised accumulators within the
    # output tolerance
    import oracle
    import int8_kv_cache_gb300 as K
    from helpers import sparse_to_device
    c = W.random_sparse(seed=S * 5 + ns, S=S, Hq=Hq, Hkv=Hkv, D=D, N=N, max_sel=max_sel,
                        invalid_frac=0.1, sigma=1.0 / 16)
    G = Hq // Hkv
    d = sparse_to_device(c)
    wsb = K.prefill_workspace_bytes(S, Hq, Hkv, D, N, max_sel, ns)
    ws = torch.full((wsb,), 255, dtype=torch.uint8, device="cuda")
    K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                  out=torch.empty_like(d["q"]), workspace=ws, num_splits=ns)
    torch.cuda.synchronize()
    blocks = -(-N // 128)
    stage = Hkv * blocks * 2 * 128 * D * 2 + S * blocks * 16 + S * 4
    off = (stage + 255) // 256 * 256
    pvec = S * Hq * ns
    f = ws[off:off + pvec * (D + 2) * 4].view(torch.float32).cpu().numpy().astype(np.float64)
    acc = f[:pvec * D].reshape(S, Hkv, ns, G, D)
    m = f[pvec * D:pvec * (D + 1)].reshape(S, Hkv, ns, G)
    l = f[pvec * (D + 1):].reshape(S, Hkv, ns, G)
    rm, rl, ra = oracle.prefill_split_partials(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                               c.scale_kind, c.idx, c.sigma, ns)
    rm = rm.reshape(S, Hkv, G, ns).transpose(0, 1, 3, 2)
    rl = rl.reshape(S, Hkv, G, ns).transpose(0, 1, 3, 2)
    ra = ra.reshape(S, Hkv, G, ns, D).transpose(0, 1, 3, 2, 4)
    live = rl > 0
    assert np.array_equal(l > 0, live)
    assert np.all(np.isneginf(m[~live]))
    bnd = np.broadcast_to(bound_of(c).reshape(S, Hkv, 1, G), (S, Hkv, ns, G))
    lse = m[live] + np.log(l[live])
    ref = rm[live] + np.log(rl[live])
    assert np.all(np.abs(lse - ref) <= bnd[live] + 1e-5 * np.abs(ref))
    on = acc[live] / l[live][:, None]
    rn = ra[live] / rl[live][:, None]
    assert np.all(np.abs(on - rn) <= 2e-3 + 1e-2 * np.abs(rn))
