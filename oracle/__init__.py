"""FP64 CPU oracle (test infrastructure only).

Import restrictions: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm use this package.  It shares no
code with ``int8_kv_cache_gb300`` and imports nothing from it.
"""
from .attention import (SCALE_PER_CHANNEL, SCALE_PER_TENSOR, apply_head_sink, attend,
                        chunk_bounds, combine, combine_all, dequantize, live_length,
                        paged_attention, paged_slots, paged_split_partials, partial,
                        sparse_attention, sparse_candidates, sparse_split_partials)
from .geometry import MODE_POW2_TILES, MODE_WAVE, split_geometry

__all__ = [
    "SCALE_PER_CHANNEL", "SCALE_PER_TENSOR", "apply_head_sink", "attend", "chunk_bounds",
    "combine", "combine_all", "dequantize", "live_length", "paged_attention", "paged_slots",
    "paged_split_partials", "partial", "sparse_attention", "sparse_candidates",
    "sparse_split_partials", "MODE_POW2_TILES", "MODE_WAVE", "split_geometry",
]
from .attention import scores, window_chunk_bounds, window_span, window_start  # noqa: E402
from .attention import e4m3fn_value  # noqa: E402
from .attention import prefill_block_ranges, prefill_split_partials  # noqa: E402
from .quantize import e4m3fn_encode, quantize_rows, quantize_rows_fp8, reshape_and_cache  # noqa

__all__ += ["quantize_rows", "reshape_and_cache", "e4m3fn_value", "e4m3fn_encode",
            "quantize_rows_fp8", "scores", "window_chunk_bounds",
            "window_span", "window_start", "prefill_block_ranges", "prefill_split_partials"]
