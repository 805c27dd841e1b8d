"""CPU oracle for the DSA hot path (Lightning Indexer + Top-K + Sparse Flash Attention).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call, link or run
anything in this package; only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares no code
with the CUDA path: it has its own FP8 codecs, its own quantisers and its own attention,
all written in numpy float64 from the definitions on the pages (cited per function).

Sources (the three pages this method is described on):

* "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient
  Inference in Kimi K3.1 Pro" -- section 1 (the DSA two-stage scheme: Lightning Indexer
  scores every historical key, Top-K filter, Sparse Flash Attention over the selected
  keys), section 2.1 (fused score + weighting + Top-K reading the paged K-cache) and
  section 2.2 (MXFP8 group-32 indexer, FP8 per-token-head-tile KV cache).
* "Adapting and Optimizing Kimi K3.1 Pro for Long-Sequence Inference" -- section 2
  (gather of the selected KV entries by index) and section 3 (hierarchical quantisation).
* "Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on Heterogeneous AI
  Hardware" -- "Lightning Indexer Three-Stream Coordination", "Full MXFP8 Quantization
  with Per-Group Dynamic Scaling for LI" (group size 32), "FP8 KVCache with
  Per-Token-Head-Tile Quantization for SFA" (tile size 128) and "Preserving a
  Mixed-Precision Path" (BF16 kept for the final attention weighting).

The pages print no formula; where they are silent the reading adopted is stated in the
function that takes it.  Pins: every function here is checked by ``tests/test_oracle_*``
against something other than itself (library codecs, closed forms, hand examples,
brute force, dense attention).  The synthetic Top-K recall diagnostic is
"parity unpinned" (the pages' recall figure needs a benchmark and trained weights).
"""

from .codecs import e4m3_decode, e4m3_encode, e8m0_decode
from .quant import (
    mxfp8_quantize,
    mxfp8_dequantize,
    fp8_tile_quantize,
    fp8_tile_dequantize,
    MX_GROUP,
    FP8_TILE,
)
from .indexer import indexer_scores_row, topk_row, indexer_topk_rows
from .sfa import sparse_attention_row
from .pipeline import decode_rows

__all__ = [
    "e4m3_decode", "e4m3_encode", "e8m0_decode",
    "mxfp8_quantize", "mxfp8_dequantize", "fp8_tile_quantize", "fp8_tile_dequantize",
    "MX_GROUP", "FP8_TILE",
    "indexer_scores_row", "topk_row", "indexer_topk_rows",
    "sparse_attention_row",
    "decode_rows",
]
