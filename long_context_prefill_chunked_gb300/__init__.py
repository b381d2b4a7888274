"""Long-context prefill attention (dense chunked + block-sparse) for one GB300 GPU.

The compute path is libpf.so (hand-written sm_103a kernels behind a C ABI,
declared in include/pf.h); ``pf`` is its thin ctypes binding.
"""
from .pf import (KeepRules, PFError, Selection, alloc_kbar, alloc_pooled, alloc_selection, attn_dense,
                 attn_indexed, attn_sparse, block_index, dense_workspace, launch_count, load,
                 set_debug_withhold, set_wait_timeout, sparse_sizes, stream_status, to_f16, vbar_view, version)

__all__ = ["KeepRules", "PFError", "Selection", "alloc_kbar", "alloc_pooled", "alloc_selection", "attn_dense",
           "attn_indexed", "attn_sparse", "block_index", "dense_workspace", "launch_count", "load",
           "set_debug_withhold", "set_wait_timeout", "sparse_sizes", "stream_status", "to_f16", "vbar_view",
           "version"]
