"""Quantize-on-write of new key / value rows into a paged INT8 cache.

TEST INFRASTRUCTURE ONLY (see ``oracle/attention.py``).

[onnxruntime PR 29912 "PagedAttention: quantized KV cache ...", CUDA kernels:
"ReshapeAndCache quantizes on write; all read paths dequantize with
k_scale/v_scale under PER_TENSOR or PER_CHANNEL granularity".]  Each new token
n has rows K_new[n, g, :], V_new[n, g, :] (fp16) and a destination slot
slot_mapping[n]; the cache row (slot, g) receives

    code[d] = clamp(round_half_even(x[d] / scale[g, d]), -127, 127)

(per-tensor: one scale).  A float8 e4m3fn cache (the schema's float8e4m3fn
element type) stores the nearest e4m3fn value of the same quotient instead,
ties to even, saturated to +-448.  Readings where the page is silent: the codes are
symmetric (-127..127, the range that dequantisation with scale = amax/127
produces); the quotient is the fp32 division of the fp16 value (widened to
fp32) by the fp32 scale, so both sides take the rounding decision in fp32; a
NaN quotient stores 0; a slot outside [0, num_slots) (padding, -1) writes
nothing.
"""
from __future__ import annotations

import math

import numpy as np

SCALE_PER_TENSOR = 1
SCALE_PER_CHANNEL = 2


def e4m3fn_encode(v: float) -> int:
    """Nearest float8 e4m3fn bit pattern of a float (ties to the even mantissa),
    saturating to +-448 (the largest finite value); NaN -> 0 (the reading taken
    for INT8 codes too).  The sign of a value that rounds to zero is kept."""
    if math.isnan(v):
        return 0
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if a >= 448.0:
        return sign | 0x7E
    # the representable magnitudes bracketing a, on the grid of a's binade
    e = max(math.frexp(a)[1] - 1, -6) if a > 0 else -6   # a in [2^e, 2^(e+1)), or subnormal
    step = 2.0 ** (e - 3)                                # 3 mantissa bits
    q = a / step                                         # exact: a power-of-two scaling
    n = math.floor(q)
    r = q - n
    if r > 0.5 or (r == 0.5 and n % 2 == 1):
        n += 1
    mag = n * step
    if mag == 0.0:
        return sign
    if mag >= 448.0:
        return sign | 0x7E
    ee = math.frexp(mag)[1] - 1
    if ee < -6:                                          # subnormal: m * 2^-9
        return sign | int(round(mag / 2.0 ** -9))
    m = int(round((mag / 2.0 ** ee - 1.0) * 8))
    return sign | ((ee + 7) << 3) | m


def quantize_rows_fp8(x: np.ndarray, scale: np.ndarray, scale_kind: int,
                      kv_head: int) -> np.ndarray:
    """float8 e4m3fn bit patterns (uint8) of rows x[..., D] of one KV head: the
    fp32 quotient x / scale, rounded to nearest even and saturated."""
    xf = np.asarray(x).astype(np.float32)
    if scale_kind == SCALE_PER_TENSOR:
        s = np.float32(np.asarray(scale, np.float32).reshape(-1)[0])
    elif scale_kind == SCALE_PER_CHANNEL:
        s = np.asarray(scale, np.float32)[kv_head]
    else:
        raise ValueError(f"unknown scale kind {scale_kind}")
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.divide(xf, s, dtype=np.float32)
    return np.array([e4m3fn_encode(float(v)) for v in q.reshape(-1)],
                    dtype=np.uint8).reshape(q.shape)


def quantize_rows(x: np.ndarray, scale: np.ndarray, scale_kind: int, kv_head: int) -> np.ndarray:
    """Codes of rows x[..., D] (fp16) of one KV head, computed in fp32."""
    xf = np.asarray(x).astype(np.float32)
    if scale_kind == SCALE_PER_TENSOR:
        s = np.float32(np.asarray(scale, np.float32).reshape(-1)[0])
    elif scale_kind == SCALE_PER_CHANNEL:
        s = np.asarray(scale, np.float32)[kv_head]
    else:
        raise ValueError(f"unknown scale kind {scale_kind}")
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(np.divide(xf, s, dtype=np.float32))
    q = np.where(np.isnan(q), np.float32(0.0), q)
    return np.clip(q, -127, 127).astype(np.int8)


def reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                      scale_kind):
    """Write the quantised rows into copies of the caches ([num_slots, Hkv, D]
    or [num_blocks, block_size, Hkv, D]; int8 caches take INT8 codes, uint8
    caches float8 e4m3fn bit patterns); returns (k_cache', v_cache')."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    shape = kc.shape
    kf = kc.reshape(-1, shape[-2], shape[-1])
    vf = vc.reshape(-1, shape[-2], shape[-1])
    num_slots, Hkv, _ = kf.shape
    enc = quantize_rows_fp8 if kc.dtype == np.uint8 else quantize_rows
    for n, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0 or slot >= num_slots:
            continue
        for g in range(Hkv):
            kf[slot, g] = enc(k_new[n, g], k_scale, scale_kind, g)
            vf[slot, g] = enc(v_new[n, g], v_scale, scale_kind, g)
    return kf.reshape(shape), vf.reshape(shape)
