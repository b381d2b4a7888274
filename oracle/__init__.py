"""Float64 CPU oracle (test infrastructure; see ``oracle.attention``).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  It shares no code with the CUDA
library and never calls it.
"""
from .attention import (MASK_DROP, KeepRules, Selection, block_counts, block_select,
                        causal_additive, chunk_kv_cache_layout, dense, dense_indexed,
                        indexed_visible_keys, pool_blocks, skip_share, sparse, sparse_for_selection,
                        tile_union)

__all__ = ["MASK_DROP", "KeepRules", "Selection", "block_counts", "block_select", "causal_additive",
           "chunk_kv_cache_layout", "dense", "dense_indexed", "indexed_visible_keys", "pool_blocks",
           "skip_share", "sparse", "sparse_for_selection", "tile_union"]
