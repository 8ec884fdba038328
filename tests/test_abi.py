"""The C ABI without a GPU: the library builds and loads, exports every symbol
that include/int8kv.h declares, its host-only geometry is bit-exact with the
oracle, and argument errors come back as status codes before any CUDA call."""
import ctypes
import itertools
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import int8_kv_cache_gb300 as K
    if not os.path.exists(K.library_path()):
        from int8_kv_cache_gb300 import build
        build.build()
    return K.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "int8kv.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*"
                                 r"([A-Za-z_][A-Za-z0-9_]*)\s*\(", src, flags=re.M)))


def test_header_declares_the_five_calls():
    names = _declared_functions()
    for n in ["dsa_decode", "dsa_prefill", "paged_decode", "split_combine", "split_geometry"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.i8kv_version() >= 100
    assert lib.i8kv_status_string(0) == b"ok"
    assert lib.i8kv_status_string(4).startswith(b"workspace")


def test_window_span_matches_the_oracle(lib):
    # host-only arithmetic: the span a windowed paged decode's splits cover
    for cap in (0, 16, 96, 512, 4096, 8192):
        for window in (-1, 0, 1, 15, 16, 80, 95, 496, 1023, 5000):
            assert lib.paged_window_span(cap, window) == oracle.window_span(cap, window)


def test_geometry_bit_exact_with_oracle(lib):
    import int8_kv_cache_gb300 as K
    caps = [0, 1, 16, 17, 64, 65, 127, 128, 129, 509, 520, 2048, 2112, 2600, 4096, 8192, 32768]
    for cap, units, wave, mode, ov in itertools.product(
            caps, [1, 2, 8, 16, 32, 128, 4096], [1, 152, 216, 304, 396, 512, 608, 1216],
            [oracle.MODE_WAVE, oracle.MODE_POW2_TILES], [0, 1, 2, 3, 128, 256, 512]):
        granule = 64 if mode == oracle.MODE_POW2_TILES else 16
        want = oracle.split_geometry(cap, units, wave, granule, 128, 32, mode, ov)
        got = K.split_geometry(cap, units, wave, granule, 128, 32, mode, ov)
        assert got == want, (cap, units, wave, mode, ov)


def test_geometry_printed_examples_through_the_abi(golden_dir):
    import json
    import int8_kv_cache_gb300 as K
    with open(os.path.join(golden_dir, "geometry_examples.json")) as f:
        for c in json.load(f)["cases"]:
            a = c["args"]
            n, chunk = K.split_geometry(a["cap"], a["units"], a["wave"], a["granule"],
                                        a["min_chunk"], a["max_splits"], a["mode"], a["override"])
            assert (n, chunk) == (c["expect"]["num_splits"], c["expect"]["chunk"]), c["name"]


def test_geometry_rejects_bad_arguments(lib):
    n, c = ctypes.c_int32(), ctypes.c_int32()
    assert lib.split_geometry(100, 0, 10, 1, 1, 32, 0, 0, ctypes.byref(n), ctypes.byref(c)) == 1
    assert lib.split_geometry(100, 1, 10, 1, 1, 32, 9, 0, ctypes.byref(n), ctypes.byref(c)) == 1
    assert lib.split_geometry(100, 1, 10, 1, 1, 32, 0, -1, ctypes.byref(n), ctypes.byref(c)) == 1
    assert lib.split_geometry(100, 1, 10, 1, 1, 32, 0, 0, None, ctypes.byref(c)) == 1


def test_workspace_bytes(lib):
    assert lib.split_workspace_bytes(16, 1, 12, 256) == 0
    assert lib.split_workspace_bytes(16, 16, 12, 256) == 16 * 16 * 12 * (256 + 2) * 4
    assert lib.split_workspace_bytes(0, 4, 4, 64) == 0


# fake, aligned, never-dereferenced device addresses: every call below must be
# rejected by host validation before any CUDA call
P = 0x10000
P8 = 0x10008


def _dsa(lib, **kw):
    a = dict(q=P, k=P, v=P, ks=P, vs=P, kind=2, idx=P, S=1, Hq=8, Hkv=2, D=128, N=100, max_sel=64,
             sigma=0.1, sink=None, ns=1, chunk=64, ws=None, wsb=0, out=P, lse=None, flags=None,
             stream=None)
    a.update(kw)
    return lib.dsa_decode(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["kind"], a["idx"], a["S"],
                          a["Hq"], a["Hkv"], a["D"], a["N"], a["max_sel"], a["sigma"], a["sink"],
                          a["ns"], a["chunk"], a["ws"], a["wsb"], a["out"], a["lse"], a["flags"],
                          a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(Hq=9), 1), (dict(Hq=36, Hkv=2), 2), (dict(sigma=2.0), 2),
    (dict(sigma=float("nan")), 1), (dict(sigma=-0.5), 1), (dict(kind=3), 1), (dict(ks=None), 1),
    (dict(q=None), 1), (dict(idx=None), 1), (dict(q=P8), 3), (dict(out=P8), 3),
    (dict(ns=33, chunk=16), 1), (dict(ns=1, chunk=48), 1), (dict(ns=1, chunk=24), 1),
    (dict(ns=2, chunk=64), 4), (dict(S=-1), 1), (dict(max_sel=-3), 1),
])
def test_dsa_decode_validation(lib, kw, status):
    assert _dsa(lib, **kw) == status


def test_paged_decode_validation(lib):
    def call(**kw):
        a = dict(q=P, k=P, v=P, dt=1, ks=P, vs=P, kind=1, bt=P, lens=P, B=2, Hq=4, Hkv=1, D=64,
                 bs=16, mb=8, nb=20, sigma=0.125, sink=None, ns=1, chunk=128, ws=None, wsb=0,
                 out=P, lse=None, slots=None, flags=None, stream=None)
        a.update(kw)
        return lib.paged_decode(a["q"], a["k"], a["v"], a["dt"], a["ks"], a["vs"], a["kind"],
                                a["bt"], a["lens"], a["B"], a["Hq"], a["Hkv"], a["D"], a["bs"],
                                a["mb"], a["nb"], a["sigma"], a["sink"], a["ns"], a["chunk"],
                                a["ws"], a["wsb"], a["out"], a["lse"], a["slots"], a["flags"],
                                a["stream"])
    assert call(bs=8) == 2
    assert call(bs=24) == 2
    assert call(dt=4) == 1
    assert call(lens=None) == 1
    assert call(ks=None) == 1
    assert call(dt=2, ks=None, vs=None, ns=2, chunk=64) == 4  # fp16 cache needs no scales
    assert call(ns=1, chunk=64) == 1  # 1 x 64 < cap 128
    assert call(sigma=1.5) == 2


def test_combine_and_convert_validation(lib):
    assert lib.split_combine(P, P, P, 4, 0, 8, 2, 128, None, P, None, None) == 1
    assert lib.split_combine(P, P, P, 4, 33, 8, 2, 128, None, P, None, None) == 1
    assert lib.split_combine(P, P, P, 4, 4, 8, 2, 100, None, P, None, None) == 2
    assert lib.int8_to_fp16(P, P, 6, None) == 1
    assert lib.int8_to_fp16(P8, P, 8, None) == 3


def test_zero_work_is_a_no_op(lib):
    # S = 0 / B = 0 / units = 0: validated, nothing enqueued, OK without a GPU
    assert _dsa(lib, S=0) == 0
    assert lib.split_combine(P, P, P, 0, 4, 8, 2, 128, None, P, None, None) == 0
    assert lib.int8_to_fp16(P, P, 0, None) == 0


def test_reshape_and_cache_validation(lib):
    def call(**kw):
        a = dict(k=P, v=P, slots=P, T=4, Hkv=2, D=64, kc=P, vc=P, ns=100, ks=P, vs=P, kind=1,
                 cd=1, flags=None, stream=None)
        a.update(kw)
        return lib.reshape_and_cache(a["k"], a["v"], a["slots"], a["T"], a["Hkv"], a["D"], a["kc"],
                                     a["vc"], a["ns"], a["ks"], a["vs"], a["kind"], a["cd"],
                                     a["flags"], a["stream"])
    assert call(D=60) == 2      # not a multiple of 8
    assert call(D=4) == 1
    assert call(T=-1) == 1
    assert call(kind=5) == 1
    assert call(slots=None) == 1
    assert call(kc=P8) == 3
    assert call(T=0) == 0       # nothing to do, nothing enqueued
    assert call(T=0, cd=3) == 0  # float8 e4m3fn cache
    assert call(cd=2) == 1      # an fp16 cache is not a quantised cache
    assert call(cd=0) == 1


def test_paged_decode_ex_validation(lib):
    def call(**kw):
        a = dict(softcap=0.0, window=-1, ns=1, chunk=512, mb=32)
        a.update(kw)
        return lib.paged_decode_ex(P, P, P, 1, P, P, 2, P, P, 0, 32, 8, 128, 16, a["mb"], 100,
                                   0.1, None, a["softcap"], a["window"], a["ns"], a["chunk"],
                                   P, 1 << 30, P, None, None, None, None)
    assert call() == 0
    assert call(softcap=-1.0) == 1
    assert call(softcap=float("nan")) == 1
    assert call(softcap=float("inf")) == 1
    assert call(window=-2) == 1
    # with a window the splits need only cover the span min(cap, window + 16)
    assert call(window=100, ns=1, chunk=112) == 1       # 112 < 116
    assert call(window=100, ns=1, chunk=128) == 0
    assert call(window=100, ns=2, chunk=64) == 0
    assert call(window=0, ns=1, chunk=16) == 0
    assert call(window=-1, ns=1, chunk=128) == 1        # no window: the cap 512
    assert call(window=5000, ns=1, chunk=496) == 1      # wide window: the cap


def test_prefill_workspace_rules(lib):
    # host arithmetic: the staged prefill's workspace is the cache as fp16
    # operand images (Hkv x ceil(N / 128) blocks x K and V x 128 x D x 2 bytes),
    # and only for the shapes the tensor-core kernel serves
    need = lib.dsa_prefill_workspace_bytes

    def stage(S, Hkv, D, N):
        # operand images, then each row's bitmask (16 bytes per 128-position
        # block) and repeat flag
        blocks = -(-N // 128)
        return Hkv * blocks * 2 * 128 * D * 2 + S * blocks * 16 + S * 4
    assert need(16, 24, 2, 256, 300, 100, 1) == stage(16, 2, 256, 300)
    assert need(2048, 24, 2, 256, 8192, 2048, 1) == stage(2048, 2, 256, 8192)
    assert need(16, 8, 2, 128, 1000, 300, 1) == stage(16, 2, 128, 1000)
    # with splits, the partials follow at the next 256-byte boundary: S x Hq x
    # splits x (D accumulators + m + l) x 4 bytes
    st = stage(16, 2, 256, 300)
    assert need(16, 24, 2, 256, 300, 100, 3) == (st + 255) // 256 * 256 + 16 * 24 * 3 * 258 * 4
    st = stage(5, 2, 128, 1000)
    assert need(5, 8, 2, 128, 1000, 300, 32) == (st + 255) // 256 * 256 + 5 * 8 * 32 * 130 * 4
    assert need(16, 24, 2, 256, 300, 100, 33) == 0   # at most 32 splits
    assert need(16, 24, 2, 256, 300, 100, -1) == 0
    assert need(16, 24, 2, 256, 3000, 100, 1) == 0   # 4 * max_sel < N: the gathering kernel
    assert need(16, 8, 2, 64, 300, 100, 1) == 0      # head_dim 64: the gathering kernel
    assert need(0, 24, 2, 256, 300, 100, 1) == 0
    assert need(16, 24, 5, 256, 300, 100, 1) == 0    # Hq not a multiple of Hkv


def test_prefill_auto_split_rule(lib):
    # host arithmetic: tiles = Hkv x ceil(S x G / 128); min(8, SMs / tiles)
    # splits where the tiles fill at most half of the SMs, else 1
    auto = lib.dsa_prefill_auto_splits
    assert auto(128, 24, 2, 152) == 6        # 24 tiles
    assert auto(2048, 24, 2, 152) == 1       # 384 tiles
    assert auto(512, 24, 2, 152) == 1        # 96 tiles: more than half the SMs
    assert auto(256, 24, 2, 152) == 3        # 48 tiles
    assert auto(16, 24, 2, 152) == 8         # 4 tiles: at most 8 splits
    assert auto(1, 2, 2, 152) == 8           # G = 1: one tile per KV head
    assert auto(640, 16, 1, 152) == 1        # 80 tiles
    assert auto(608, 16, 1, 152) == 2        # 76 tiles: exactly half
    for S in range(1, 3000, 37):
        for G, Hkv in ((12, 2), (16, 1), (1, 8), (4, 4)):
            tiles = Hkv * -(-S * G // 128)
            want = min(8, 152 // tiles) if 2 * tiles <= 152 else 1
            assert auto(S, G * Hkv, Hkv, 152) == want, (S, G, Hkv)
    assert auto(0, 24, 2, 152) == 0 and auto(16, 24, 2, 0) == 0 and auto(16, 24, 5, 152) == 0


def test_prefill_workspace_errors_before_any_launch(lib):
    # checked before anything touches the device: the addresses are never read
    fake = 1 << 20
    args = [fake, fake, fake, fake, fake, 2, fake, 16, 24, 2, 256, 300, 100, 1.0 / 16, None]
    tail = [fake, None, None, None]
    need = lib.dsa_prefill_workspace_bytes(16, 24, 2, 256, 300, 100, 1)
    assert lib.dsa_prefill_ws(*args, 1, fake, need - 16, *tail) == 4   # I8KV_EWORKSPACE
    assert lib.dsa_prefill_ws(*args, 1, fake + 8, need, *tail) == 3    # I8KV_EALIGN
    # splits: their partials must fit too, and need a workspace
    need3 = lib.dsa_prefill_workspace_bytes(16, 24, 2, 256, 300, 100, 3)
    assert lib.dsa_prefill_ws(*args, 3, fake, need, *tail) == 4
    assert lib.dsa_prefill_ws(*args, 3, fake, need3 - 16, *tail) == 4
    assert lib.dsa_prefill_ws(*args, 3, None, 0, *tail) == 4
    assert lib.dsa_prefill_ws(*args, 33, fake, need3, *tail) == 1     # I8KV_EINVAL
    assert lib.dsa_prefill_ws(*args, -1, fake, need3, *tail) == 1
