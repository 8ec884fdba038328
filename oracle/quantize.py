"""Quantize-on-write of new key / value rows into a paged INT8 cache.

TEST INFRASTRUCTURE ONLY (see ``oracle/attention.py``).

[onnxruntime PR 29912 "PagedAttention: quantized KV cache ...", CUDA kernels:
"ReshapeAndCache quantizes on write; all read paths dequantize with
k_scale/v_scale under PER_TENSOR or PER_CHANNEL granularity".]  Each new token
n has rows K_new[n, g, :], V_new[n, g, :] (fp16) and a destination slot
slot_mapping[n]; the cache row (slot, g) receives

    code[d] = clamp(round_half_even(x[d] / scale[g, d]), -127, 127)

(per-tensor: one scale).  Readings where the page is silent: the codes are
symmetric (-127..127, the range that dequantisation with scale = amax/127
produces); the quotient is the fp32 division of the fp16 value (widened to
fp32) by the fp32 scale, so both sides take the rounding decision in fp32; a
NaN quotient stores 0; a slot outside [0, num_slots) (padding, -1) writes
nothing.
"""
from __future__ import annotations

import numpy as np

SCALE_PER_TENSOR = 1
SCALE_PER_CHANNEL = 2


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
    or [num_blocks, block_size, Hkv, D]); returns (k_cache', v_cache')."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    shape = kc.shape
    kf = kc.reshape(-1, shape[-2], shape[-1])
    vf = vc.reshape(-1, shape[-2], shape[-1])
    num_slots, Hkv, _ = kf.shape
    for n, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0 or slot >= num_slots:
            continue
        for g in range(Hkv):
            kf[slot, g] = quantize_rows(k_new[n, g], k_scale, scale_kind, g)
            vf[slot, g] = quantize_rows(v_new[n, g], v_scale, scale_kind, g)
    return kf.reshape(shape), vf.reshape(shape)
