"""Split geometry: number of splits and chunk length from the capacity and the
row count alone (never from a live sequence length).

TEST INFRASTRUCTURE ONLY (see ``oracle/attention.py``).  This is the plain
restatement the host library's ``split_geometry`` is compared with, bit for bit.

Two rules from the pages:

* WAVE rule  [onnx-genai PR 1350 "adaptive split-KV sizing", Summary]:
    target     = ceil(TARGET_BLOCKS / rows)
    num_splits = min(target, ceil(cap / MIN_CHUNK), MAX_SPLITS)
    chunk      = ceil(cap / num_splits)
  TARGET_BLOCKS is one occupancy wave of resident CTAs (here: ``wave``, the
  SM count times the kernel's resident CTAs per SM).  ``rows`` counts grid
  rows; the grid here spans KV heads too, so ``units`` = rows x kv_heads.
  A positive ``override`` pins a fixed chunk instead (the page's
  ONNX_GENAI_ATTN_SPLIT_CHUNK, "reproduces pre-adaptive behaviour"):
  num_splits = min(ceil(cap / override), MAX_SPLITS).

* POW2_TILES rule  [onnxruntime PR 33707, Summary of Changes §2,
  GetInt8TcDecodeSplitCount]: tiles = ceil(cap / granule) (64-candidate
  tiles); tiles_per_split is the smallest power of two for which
  ceil(tiles / tps) * units fits one wave; num_splits = ceil(tiles / tps), at
  most MAX_SPLITS (32); a positive ``override`` is a tiles-per-split *target*
  to which the cap and the even distribution still apply.

Readings where the pages leave a step open:

* "even distribution of a row's tiles" = tiles_eff = ceil(tiles / num_splits);
  split k covers tiles [k*tiles_eff, (k+1)*tiles_eff); the split count is then
  recomputed as ceil(tiles / tiles_eff) so that no launched split is empty by
  construction (8192 candidates at 1 tile per split -> 32 splits of 4 tiles).
* WAVE rule with ``granule`` > 1: the chunk is rounded up to a multiple of
  the granule and the split count recomputed as ceil(cap / chunk); granule 1
  reproduces the page's formula exactly.
* cap <= 0 gives one split of one granule.
* MAX_SPLITS is not stated on the onnx-genai page; 32 is taken from the
  onnxruntime page ("at most 32").
"""
from __future__ import annotations

MODE_WAVE = 0
MODE_POW2_TILES = 1


def ceil_div(a: int, b: int) -> int:
    return -((-a) // b)


def split_geometry(cap: int, units: int, wave: int, granule: int, min_chunk: int,
                   max_splits: int, mode: int, override: int = 0):
    """Return (num_splits, chunk) as Python ints."""
    if units < 1 or wave < 1 or granule < 1 or min_chunk < 1 or max_splits < 1 or override < 0:
        raise ValueError("invalid geometry arguments")
    if cap <= 0:
        return 1, granule
    if mode == MODE_WAVE:
        if override > 0:
            n = min(ceil_div(cap, override), max_splits)
        else:
            target = ceil_div(wave, units)
            n = min(target, ceil_div(cap, min_chunk), max_splits)
        n = max(n, 1)
        chunk = ceil_div(cap, n)
        chunk = ceil_div(chunk, granule) * granule
        return ceil_div(cap, chunk), chunk
    if mode == MODE_POW2_TILES:
        tiles = ceil_div(cap, granule)
        if override > 0:
            tps = override
        else:
            tps = 1
            while ceil_div(tiles, tps) * units > wave and tps < tiles:
                tps *= 2
        n = max(1, min(ceil_div(tiles, tps), max_splits))
        tiles_eff = ceil_div(tiles, n)
        return ceil_div(tiles, tiles_eff), tiles_eff * granule
    raise ValueError(f"unknown geometry mode {mode}")
