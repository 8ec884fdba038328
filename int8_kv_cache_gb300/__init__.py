"""Python binding of ``libint8kv.so``: split-KV GQA decode attention over an
INT8-quantized KV cache on GB300.

Every function here has the name and the meaning of the C entry point of the
same name in ``include/int8kv.h``.  The binding only marshals arguments: it
reads shapes from the tensors, checks dtype / device / contiguity, passes raw
device pointers and the current CUDA stream, and turns a non-zero status into
an exception.  All computation runs in the library's CUDA kernels; there is
no fallback.  PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "Int8KVError", "load", "library_path", "split_geometry", "split_workspace_bytes",
    "decode_plan", "dsa_decode", "dsa_prefill", "prefill_workspace_bytes", "paged_decode", "split_combine", "int8_to_fp16",
    "dsa_decode_static_workspace", "STATIC_WORKSPACE_BYTES", "reshape_and_cache",
    "FLAG_BAD_SLOT", "FLAG_FP32_PATH", "FLAG_WAIT_TIMEOUT", "paged_decode_ex", "window_span",
    "CACHE_FP8", "fp8_to_fp16",
    "SCALE_PER_TENSOR", "SCALE_PER_CHANNEL", "CACHE_INT8", "CACHE_FP16", "GEOM_WAVE",
    "GEOM_POW2_TILES", "GEOM_BALANCED", "PATH_DSA", "PATH_PAGED", "MAX_SPLITS", "FLAG_LEN_CLAMPED",
    "FLAG_QUERY_RANGE", "FLAG_BAD_BLOCK",
]

SCALE_PER_TENSOR = 1
SCALE_PER_CHANNEL = 2
CACHE_INT8 = 1
CACHE_FP16 = 2
CACHE_FP8 = 3
GEOM_WAVE = 0
GEOM_POW2_TILES = 1
GEOM_BALANCED = 2
PATH_DSA = 1
PATH_PAGED = 2
MAX_SPLITS = 32
FLAG_LEN_CLAMPED = 0x1
FLAG_QUERY_RANGE = 0x2
FLAG_BAD_BLOCK = 0x4
FLAG_BAD_SLOT = 0x8
FLAG_FP32_PATH = 0x10
FLAG_WAIT_TIMEOUT = 0x20
STATIC_WORKSPACE_BYTES = 4 * 1024 * 1024

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB: Optional[ctypes.CDLL] = None

_c_i32, _c_i64, _c_f32, _c_sz, _c_vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                        ctypes.c_size_t, ctypes.c_void_p)
_P_I32 = ctypes.POINTER(ctypes.c_int32)
_P_SZ = ctypes.POINTER(ctypes.c_size_t)

_SIGNATURES = {
    "i8kv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "i8kv_version": (_c_i32, []),
    "i8kv_last_cuda_error": (_c_i32, []),
    "paged_window_span": (_c_i64, [_c_i64, _c_i32]),
    "split_geometry": (_c_i32, [_c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                _P_I32, _P_I32]),
    "split_workspace_bytes": (_c_sz, [_c_i32, _c_i32, _c_i32, _c_i32]),
    "decode_plan": (_c_i32, [_c_i32, _c_i32, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                             _c_i32, _P_I32, _P_I32, _P_SZ, _P_I32]),
    "dsa_decode": (_c_i32, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i32, _c_vp, _c_i32, _c_i32,
                            _c_i32, _c_i32, _c_i64, _c_i32, _c_f32, _c_vp, _c_i32, _c_i32, _c_vp,
                            _c_sz, _c_vp, _c_vp, _c_vp, _c_vp]),
    "dsa_prefill": (_c_i32, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i32, _c_vp, _c_i32, _c_i32,
                             _c_i32, _c_i32, _c_i64, _c_i32, _c_f32, _c_vp, _c_vp, _c_vp, _c_vp,
                             _c_vp]),
    "dsa_prefill_workspace_bytes": (_c_sz, [_c_i32, _c_i32, _c_i32, _c_i32, _c_i64, _c_i32,
                                            _c_i32]),
    "dsa_prefill_auto_splits": (_c_i32, [_c_i32, _c_i32, _c_i32, _c_i32]),
    "dsa_prefill_ws": (_c_i32, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i32, _c_vp, _c_i32, _c_i32,
                                _c_i32, _c_i32, _c_i64, _c_i32, _c_f32, _c_vp, _c_i32, _c_vp,
                                _c_sz, _c_vp, _c_vp, _c_vp, _c_vp]),
    "paged_decode": (_c_i32, [_c_vp, _c_vp, _c_vp, _c_i32, _c_vp, _c_vp, _c_i32, _c_vp, _c_vp,
                              _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i64, _c_f32,
                              _c_vp, _c_i32, _c_i32, _c_vp, _c_sz, _c_vp, _c_vp, _c_vp, _c_vp,
                              _c_vp]),
    "paged_decode_ex": (_c_i32, [_c_vp, _c_vp, _c_vp, _c_i32, _c_vp, _c_vp, _c_i32, _c_vp,
                                 _c_vp, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i64,
                                 _c_f32, _c_vp, _c_f32, _c_i32, _c_i32, _c_i32, _c_vp, _c_sz,
                                 _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "split_combine": (_c_i32, [_c_vp, _c_vp, _c_vp, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                               _c_vp, _c_vp, _c_vp, _c_vp]),
    "int8_to_fp16": (_c_i32, [_c_vp, _c_vp, _c_i64, _c_vp]),
    "reshape_and_cache": (_c_i32, [_c_vp, _c_vp, _c_vp, _c_i32, _c_i32, _c_i32, _c_vp, _c_vp,
                                   _c_i64, _c_vp, _c_vp, _c_i32, _c_i32, _c_vp, _c_vp]),
    "fp8_to_fp16": (_c_i32, [_c_vp, _c_vp, _c_i64, _c_vp]),
    "dsa_decode_static_workspace": (_c_i32, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i32, _c_vp,
                                             _c_i32, _c_i32, _c_i32, _c_i32, _c_i64, _c_i32,
                                             _c_f32, _c_vp, _c_i32, _c_i32, _c_vp, _c_vp, _c_vp,
                                             _c_vp]),
}


class Int8KVError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        msg = f"{fn}: {load().i8kv_status_string(status).decode()} (status {status})"
        if detail:
            msg += f"; {detail}"
        super().__init__(msg)


def library_path() -> str:
    return os.path.join(_HERE, "libint8kv.so")


def load() -> ctypes.CDLL:
    """Load the in-tree library (build it with ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(fn: str, status: int):
    if status != 0:
        detail = ""
        if status == 5:
            detail = f"cudaError {load().i8kv_last_cuda_error()}"
        raise Int8KVError(fn, status, detail)


def _t(x: Optional[torch.Tensor], dtype, name: str) -> Optional[int]:
    """Device pointer of a contiguous CUDA tensor of the given dtype (None -> NULL)."""
    if x is None:
        return None
    try:
        ok = (dtype is None or x.dtype == dtype or
              (type(dtype) is tuple and x.dtype in dtype)) and x.is_cuda and x.is_contiguous()
    except AttributeError:
        raise TypeError(f"{name} must be a torch.Tensor") from None
    if not ok:
        if dtype is not None and x.dtype != dtype and not (type(dtype) is tuple and
                                                           x.dtype in dtype):
            raise TypeError(f"{name}: expected {dtype}, got {x.dtype}")
        if not x.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        raise ValueError(f"{name} must be contiguous")
    return x.data_ptr()


def _on_current_device(x: torch.Tensor, name: str) -> None:
    """The library works on the current CUDA device (its kernels, its cached
    launch attributes and its static workspace are per device): refuse tensors
    that live on another one."""
    if x.is_cuda and x.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {x.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}; call under "
                         f"torch.cuda.device({x.device})")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# --------------------------------------------------------------------------
# host-only calls
# --------------------------------------------------------------------------

def split_geometry(cap: int, units: int, wave_ctas: int, granule: int, min_chunk: int,
                   max_splits: int, mode: int, override_value: int = 0):
    """(num_splits, chunk) -- pure host integer arithmetic in the library."""
    n, c = ctypes.c_int32(), ctypes.c_int32()
    _check("split_geometry", load().split_geometry(cap, units, wave_ctas, granule, min_chunk,
                                                   max_splits, mode, override_value,
                                                   ctypes.byref(n), ctypes.byref(c)))
    return n.value, c.value


def split_workspace_bytes(units: int, num_splits: int, G: int, D: int) -> int:
    return int(load().split_workspace_bytes(units, num_splits, G, D))


def decode_plan(path: int, cache_dtype: int, cap: int, rows: int, Hq: int, Hkv: int, D: int,
                mode: int, override_value: int = 0):
    """(num_splits, chunk, workspace_bytes, wave_ctas) on the current device."""
    n, c, w = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    ws = ctypes.c_size_t()
    _check("decode_plan", load().decode_plan(path, cache_dtype, cap, rows, Hq, Hkv, D, mode,
                                             override_value, ctypes.byref(n), ctypes.byref(c),
                                             ctypes.byref(ws), ctypes.byref(w)))
    return n.value, c.value, int(ws.value), w.value


# --------------------------------------------------------------------------
# device calls
# --------------------------------------------------------------------------

def dsa_decode(q, k_cache, v_cache, k_scale, v_scale, scale_kind: int, idx,
               softmax_scale: float, head_sink=None, num_splits: int = 0, chunk: int = 0,
               workspace=None, out=None, lse=None, flags=None, stream=None,
               partials_only: bool = False):
    """Sparse-candidate decode.  q [S, Hq, D] fp16; caches [N, Hkv, D] int8;
    idx [S, max_sel] int32.  Returns ``out`` ([S, Hq, D] fp16).  With
    ``partials_only`` (and num_splits > 1) only the workspace partials are
    written (out is NULL at the C ABI) and None is returned."""
    _on_current_device(q, "q")
    S, Hq, D = q.shape
    N, Hkv, _ = k_cache.shape
    max_sel = idx.shape[1]
    if out is None and not partials_only:
        out = torch.empty_like(q)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("dsa_decode", load().dsa_decode(
        _t(q, torch.float16, "q"), _t(k_cache, torch.int8, "k_cache"),
        _t(v_cache, torch.int8, "v_cache"), _t(k_scale, torch.float32, "k_scale"),
        _t(v_scale, torch.float32, "v_scale"), scale_kind, _t(idx, torch.int32, "idx"), S, Hq,
        Hkv, D, N, max_sel, softmax_scale, _t(head_sink, torch.float32, "head_sink"), num_splits,
        chunk, _t(workspace, None, "workspace"), ws_bytes, _t(out, torch.float16, "out"),
        _t(lse, torch.float32, "lse"), _t(flags, torch.int32, "flags"), _stream(stream)))
    return out


def prefill_workspace_bytes(S: int, Hq: int, Hkv: int, D: int, N: int, max_sel: int,
                            num_splits: int = 0) -> int:
    """Bytes of the workspace that gives dsa_prefill the staged tensor-core form
    for this shape and split count (the library's dsa_prefill_workspace_bytes;
    0 where that kernel does not serve the shape)."""
    return int(load().dsa_prefill_workspace_bytes(S, Hq, Hkv, D, N, max_sel, num_splits))


def dsa_prefill(q, k_cache, v_cache, k_scale, v_scale, scale_kind: int, idx,
                softmax_scale: float, head_sink=None, out=None, lse=None, flags=None,
                stream=None, workspace=None, num_splits: int = 0):
    """Sparse-candidate prefill.  With a workspace (a device tensor of
    prefill_workspace_bytes(..., num_splits) bytes or more) the call takes
    dsa_prefill_ws: the cache is converted once into fp16 operand images
    there, and with num_splits (0: automatic) each tile's blocks may be split
    over several CTAs whose partials the combine kernel merges."""
    _on_current_device(q, "q")
    S, Hq, D = q.shape
    N, Hkv, _ = k_cache.shape
    max_sel = idx.shape[1]
    if out is None:
        out = torch.empty_like(q)
    args = (_t(q, torch.float16, "q"), _t(k_cache, torch.int8, "k_cache"),
            _t(v_cache, torch.int8, "v_cache"), _t(k_scale, torch.float32, "k_scale"),
            _t(v_scale, torch.float32, "v_scale"), scale_kind, _t(idx, torch.int32, "idx"), S,
            Hq, Hkv, D, N, max_sel, softmax_scale, _t(head_sink, torch.float32, "head_sink"))
    tail = (_t(out, torch.float16, "out"), _t(lse, torch.float32, "lse"),
            _t(flags, torch.int32, "flags"), _stream(stream))
    if workspace is None and num_splits == 0:
        _check("dsa_prefill", load().dsa_prefill(*args, *tail))
    else:
        if workspace is not None:
            _on_current_device(workspace, "workspace")
        _check("dsa_prefill_ws", load().dsa_prefill_ws(
            *args, num_splits, _t(workspace, None, "workspace"),
            0 if workspace is None else workspace.numel() * workspace.element_size(), *tail))
    return out


def window_span(cap: int, window: int) -> int:
    """Positions the splits of a windowed paged decode cover (the library's
    paged_window_span, i.e. I8KV_WINDOW_SPAN)."""
    return int(load().paged_window_span(cap, window))


def paged_decode(q, k_cache, v_cache, k_scale, v_scale, scale_kind: int, block_table, seq_lens,
                 softmax_scale: float, head_sink=None, num_splits: int = 0, chunk: int = 0,
                 workspace=None, out=None, lse=None, slots_out=None, flags=None, stream=None,
                 partials_only: bool = False, softcap: float = 0.0, window: int = -1):
    """Paged decode.  q [B, Hq, D] fp16; caches [num_blocks, block_size, Hkv, D]
    int8 or fp16; block_table [B, max_blocks] int32; seq_lens [B] int32 (device).
    With ``partials_only`` (and num_splits > 1) only the workspace partials are
    written and None is returned.  ``softcap`` > 0 or ``window`` >= 0 go through
    the C entry point paged_decode_ex, the defaults through paged_decode."""
    _on_current_device(q, "q")
    B, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    max_blocks = block_table.shape[1]
    cache_dtype = _cache_dtype(k_cache)
    if out is None and not partials_only:
        out = torch.empty_like(q)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    head = (_t(q, torch.float16, "q"), _t(k_cache, k_cache.dtype, "k_cache"),
            _t(v_cache, k_cache.dtype, "v_cache"), cache_dtype,
            _t(k_scale, torch.float32, "k_scale"), _t(v_scale, torch.float32, "v_scale"),
            scale_kind, _t(block_table, torch.int32, "block_table"),
            _t(seq_lens, torch.int32, "seq_lens"), B, Hq, Hkv, D, bs, max_blocks, nb,
            softmax_scale, _t(head_sink, torch.float32, "head_sink"))
    tail = (num_splits, chunk, _t(workspace, None, "workspace"), ws_bytes,
            _t(out, torch.float16, "out"), _t(lse, torch.float32, "lse"),
            _t(slots_out, torch.int32, "slots_out"), _t(flags, torch.int32, "flags"),
            _stream(stream))
    if softcap == 0.0 and window == -1:
        _check("paged_decode", load().paged_decode(*head, *tail))
    else:
        _check("paged_decode_ex", load().paged_decode_ex(*head, float(softcap), int(window),
                                                         *tail))
    return out


def paged_decode_ex(*args, softcap: float = 0.0, window: int = -1, **kw):
    """paged_decode with the softcap / sliding-window options (same arguments)."""
    return paged_decode(*args, softcap=softcap, window=window, **kw)


def split_combine(acc, m, l, Hq: int, Hkv: int, head_sink=None, out=None, lse=None,
                  stream=None):
    """Combine partials acc [units, splits, G, D], m, l [units, splits, G] (fp32)."""
    _on_current_device(acc, "acc")
    units, ns, G, D = acc.shape
    if out is None:
        out = torch.empty((units * G, D), dtype=torch.float16, device=acc.device)
    _check("split_combine", load().split_combine(
        _t(acc, torch.float32, "acc"), _t(m, torch.float32, "m"), _t(l, torch.float32, "l"),
        units, ns, Hq, Hkv, D, _t(head_sink, torch.float32, "head_sink"),
        _t(out, torch.float16, "out"), _t(lse, torch.float32, "lse"), _stream(stream)))
    return out


def _cache_dtype(t, allow_fp16=True):
    """The C cache-dtype code of a cache tensor: int8 -> INT8, float8_e4m3fn or
    uint8 (e4m3fn bit patterns) -> FP8, float16 -> FP16."""
    if t.dtype == torch.int8:
        return CACHE_INT8
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return CACHE_FP8
    if allow_fp16 and t.dtype == torch.float16:
        return CACHE_FP16
    raise TypeError(f"unsupported cache dtype {t.dtype}")


def reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                      scale_kind: int, flags=None, stream=None):
    """Quantize new rows k_new / v_new [T, Hkv, D] (fp16) into the INT8 or
    float8 e4m3fn caches (int8, or uint8 / float8_e4m3fn tensors, [num_slots,
    Hkv, D] or [num_blocks, block_size, Hkv, D]) at slot_mapping [T]."""
    _on_current_device(k_new, "k_new")
    T, Hkv, D = k_new.shape
    num_slots = k_cache.numel() // (Hkv * D)
    cd = _cache_dtype(k_cache, allow_fp16=False)
    _check("reshape_and_cache", load().reshape_and_cache(
        _t(k_new, torch.float16, "k_new"), _t(v_new, torch.float16, "v_new"),
        _t(slot_mapping, torch.int32, "slot_mapping"), T, Hkv, D,
        _t(k_cache, k_cache.dtype, "k_cache"), _t(v_cache, k_cache.dtype, "v_cache"), num_slots,
        _t(k_scale, torch.float32, "k_scale"), _t(v_scale, torch.float32, "v_scale"), scale_kind,
        cd, _t(flags, torch.int32, "flags"), _stream(stream)))


def fp8_to_fp16(x, out=None, stream=None):
    """The paged decode kernel's float8 e4m3fn -> fp16 conversion over a uint8
    buffer of e4m3fn bit patterns (n % 4 == 0)."""
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    _check("fp8_to_fp16", load().fp8_to_fp16(_t(x, x.dtype, "x"), _t(out, torch.float16, "out"),
                                             x.numel(), _stream(stream)))
    return out


def int8_to_fp16(x, out=None, stream=None):
    """The decode kernels' int8 -> fp16 conversion over a buffer (n % 4 == 0)."""
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    _check("int8_to_fp16", load().int8_to_fp16(_t(x, torch.int8, "x"),
                                               _t(out, torch.float16, "out"), x.numel(),
                                               _stream(stream)))
    return out


def dsa_decode_static_workspace(q, k_cache, v_cache, k_scale, v_scale, scale_kind: int, idx,
                                softmax_scale: float, head_sink=None, num_splits: int = 0,
                                chunk: int = 0, out=None, lse=None, flags=None, stream=None):
    """dsa_decode with the split partials in the library's own fixed device
    array (STATIC_WORKSPACE_BYTES), for callers that cannot allocate scratch
    memory when they call; calls that may run concurrently on the GPU must not
    use it (they share the array)."""
    _on_current_device(q, "q")
    S, Hq, D = q.shape
    N, Hkv, _ = k_cache.shape
    max_sel = idx.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _check("dsa_decode_static_workspace", load().dsa_decode_static_workspace(
        _t(q, torch.float16, "q"), _t(k_cache, torch.int8, "k_cache"),
        _t(v_cache, torch.int8, "v_cache"), _t(k_scale, torch.float32, "k_scale"),
        _t(v_scale, torch.float32, "v_scale"), scale_kind, _t(idx, torch.int32, "idx"), S, Hq,
        Hkv, D, N, max_sel, softmax_scale, _t(head_sink, torch.float32, "head_sink"), num_splits,
        chunk, _t(out, torch.float16, "out"), _t(lse, torch.float32, "lse"),
        _t(flags, torch.int32, "flags"), _stream(stream)))
    return out
