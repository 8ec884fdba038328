"""Shared test plumbing: move a workload case to the GPU, run the CUDA path
through the binding, and compare with the FP64 oracle."""
import math

import numpy as np
import torch

import int8_kv_cache_gb300 as K
import oracle

# Elementwise bar for fp16 outputs against the FP64 oracle: the stated
# "max abs <= 2e-3, max rel <= 1e-2" read as |gpu - ref| <= 2e-3 + 1e-2 |ref|.
ATOL, RTOL = 2e-3, 1e-2
# split vs unsplit: |a - b| <= 1e-3 * max(1, |b|); lse to 1e-4 absolute
SPLIT_TOL, LSE_TOL = 1e-3, 1e-4


def dev(x, dtype=None):
    if x is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def sparse_to_device(c):
    return dict(q=dev(c.q), k=dev(c.k_codes), v=dev(c.v_codes), ks=dev(c.k_scale),
                vs=dev(c.v_scale), idx=dev(c.idx), sink=dev(c.sink))


def paged_to_device(c):
    return dict(q=dev(c.q), k=dev(c.k_cache), v=dev(c.v_cache), ks=dev(c.k_scale),
                vs=dev(c.v_scale), bt=dev(c.block_table), lens=dev(c.seq_lens), sink=dev(c.sink))


def _unpack_partials(ws, units, ns, G, D):
    """Workspace floats -> (m, l [units, ns, G], acc [units, ns, G, D]) float64."""
    w = ws.cpu().numpy().astype(np.float64)
    n = units * ns * G
    acc = w[:n * D].reshape(units, ns, G, D)
    m = w[n * D:n * (D + 1)].reshape(units, ns, G)
    l = w[n * (D + 1):n * (D + 2)].reshape(units, ns, G)
    return m, l, acc


def run_dsa(c, d=None, num_splits=0, chunk=0, prefill=False, flags=None, partials=False,
            staged=False):
    """Sparse decode (or prefill) through the binding: (O, lse) as float64, or
    with ``partials`` the workspace partials of a partials-only decode call.
    ``staged``: the prefill with a workspace (filled with 0xFF bytes first),
    its tensor-core path split ``num_splits`` ways (0: automatic)."""
    d = d or sparse_to_device(c)
    S, Hq, D = c.q.shape
    Hkv = c.k_codes.shape[1]
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device="cuda")
    if prefill:
        ws = None
        if staged:
            wsb = K.prefill_workspace_bytes(S, Hq, Hkv, D, c.k_codes.shape[0], c.idx.shape[1],
                                            num_splits)
            ws = torch.full((max(wsb, 16),), 255, dtype=torch.uint8, device="cuda")
        K.dsa_prefill(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                      d["sink"], out=out, lse=lse, flags=flags, workspace=ws,
                      num_splits=num_splits if staged else 0)
    else:
        ns = num_splits
        if ns == 0:
            ns, chunk, wsb, _ = K.decode_plan(K.PATH_DSA, K.CACHE_INT8, c.idx.shape[1], S, Hq, Hkv,
                                              D, K.GEOM_POW2_TILES, 0)
        wsb = K.split_workspace_bytes(S * Hkv, ns, Hq // Hkv, D)
        ws = torch.full((max(wsb // 4, 1),), float("nan"), dtype=torch.float32, device="cuda")
        K.dsa_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["idx"], c.sigma,
                     d["sink"], num_splits=ns, chunk=chunk, workspace=ws,
                     out=None if partials else out, lse=None if partials else lse, flags=flags,
                     partials_only=partials)
        if partials:
            torch.cuda.synchronize()
            return _unpack_partials(ws, S * Hkv, ns, Hq // Hkv, D)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def run_paged(c, d=None, num_splits=0, chunk=0, slots=False, flags=None, softcap=0.0,
              window=-1, partials=False):
    """Paged decode through the binding.  Returns (O, lse[, slots]) as float64
    arrays, or with ``partials`` the workspace partials (m, l [units, ns, G],
    acc [units, ns, G, D]) of a partials-only call."""
    d = d or paged_to_device(c)
    B, Hq, D = c.q.shape
    nb, bs, Hkv, _ = c.k_cache.shape
    G = Hq // Hkv
    cap = c.block_table.shape[1] * bs
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ns = num_splits
    if ns == 0:
        dt = {np.dtype(np.float16): K.CACHE_FP16, np.dtype(np.uint8): K.CACHE_FP8}.get(
            c.k_cache.dtype, K.CACHE_INT8)
        ns, chunk, _, _ = K.decode_plan(K.PATH_PAGED, dt, K.window_span(cap, window), B, Hq, Hkv,
                                        D, K.GEOM_WAVE, 0)
    wsb = K.split_workspace_bytes(B * Hkv, ns, G, D)
    ws = torch.full((max(wsb // 4, 1),), float("nan"), dtype=torch.float32, device="cuda")
    so = torch.full((B, cap), -99, dtype=torch.int32, device="cuda") if slots else None
    K.paged_decode(d["q"], d["k"], d["v"], d["ks"], d["vs"], c.scale_kind, d["bt"], d["lens"],
                   c.sigma, d["sink"], num_splits=ns, chunk=chunk, workspace=ws,
                   out=None if partials else out, lse=None if partials else lse, slots_out=so,
                   flags=flags, partials_only=partials, softcap=softcap, window=window)
    torch.cuda.synchronize()
    if partials:
        return _unpack_partials(ws, B * Hkv, ns, G, D)
    res = (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))
    if slots:
        res = res + (so.cpu().numpy(),)
    return res


def oracle_dsa(c):
    return oracle.sparse_attention(c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale, c.scale_kind,
                                   c.idx, c.sigma, c.sink)


def oracle_paged(c, softcap=0.0, window=-1):
    return oracle.paged_attention(c.q, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.scale_kind,
                                  c.block_table, c.seq_lens, c.sigma, c.sink, softcap=softcap,
                                  window=window)


def assert_close_oracle(got, ref, what=""):
    """fp16 outputs against the FP64 oracle, elementwise."""
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r}")


def lse_bound(q, k_scale, scale_kind, Hkv, sigma, fp16_cache=False, code_max=128.0):
    """Per (row, head) bound on |lse_gpu - lse_ref| from folding k_scale into an
    fp16 query: eps = sigma * code_max * sum_d |Q'_d - fp16(Q'_d)|, Q' =
    fp32(Q * k_scale) (the error budget of onnxruntime PR 33707 §1; code_max
    bounds |code|: 128 for INT8, 448 for float8 e4m3fn), plus 1e-5 for fp32 /
    exp2 rounding.  Shape [rows, Hq]."""
    R, Hq, D = q.shape
    G = Hq // Hkv
    if fp16_cache:
        return np.full((R, Hq), 1e-5)
    qf = q.astype(np.float32)
    if scale_kind == 1:
        ks = np.broadcast_to(np.float32(k_scale.reshape(-1)[0]), (Hq, D))
    else:
        ks = np.repeat(k_scale.astype(np.float32), G, axis=0)  # [Hq, D]
    qp = (qf * ks[None]).astype(np.float32)
    rnd = np.abs(qp.astype(np.float64) - qp.astype(np.float16).astype(np.float64))
    return sigma * code_max * rnd.sum(axis=-1) + 1e-5


def assert_lse_oracle(got, ref, bound, what=""):
    """lse against the oracle within the per-head query-rounding bound."""
    assert np.all(np.isneginf(got) == np.isneginf(ref)), f"{what}: -inf pattern differs"
    fin = ~np.isneginf(ref)
    err = np.abs(got[fin] - ref[fin])
    b = bound[fin] + 1e-6 * np.abs(ref[fin])
    assert np.all(err <= b), f"{what}: lse err {err.max()} above bound (worst ratio " \
                             f"{(err / b).max():.3f})"


def assert_lse_close(got, ref, tol=1e-4, what=""):
    both_inf = np.isneginf(got) & np.isneginf(ref)
    fin = ~both_inf
    assert np.all(np.isneginf(got) == np.isneginf(ref)), f"{what}: -inf pattern differs"
    if np.any(fin):
        err = np.abs(got[fin] - ref[fin])
        assert np.all(err <= tol * np.maximum(1.0, np.abs(ref[fin]))), \
            f"{what}: lse max err {err.max()}"


def assert_split_close(a, b, what=""):
    err = np.abs(a - b)
    assert np.all(err <= SPLIT_TOL * np.maximum(1.0, np.abs(b))), \
        f"{what}: split vs unsplit max err {err.max()}"


def paged_bound(c):
    """lse tolerance of a paged case (int8, float8 e4m3fn or fp16 cache)."""
    return lse_bound(c.q, c.k_scale, c.scale_kind, c.k_cache.shape[2], c.sigma,
                     fp16_cache=c.k_cache.dtype == np.float16,
                     code_max=448.0 if c.k_cache.dtype == np.uint8 else 128.0)
