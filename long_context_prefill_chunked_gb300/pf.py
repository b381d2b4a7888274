"""Python binding of libpf (ctypes): argument marshalling only.

Every computation runs in libpf's CUDA kernels; PyTorch provides device
memory and the stream.  Functions mirror the C ABI in include/pf.h:

    attn_dense(q, k_hist, v_hist, k_chunk, v_chunk, start_pos, mask=None, ...)
    block_index(q, k, start_pos, block=128, alpha=0.1, sel=None)
    attn_sparse(q, k, v, start_pos, sel, block=128, pooled=None, out=None)

Tensors are token-major with the head dim contiguous: q [B, C, Hq, d],
k_hist/v_hist [B, start_pos, Hkv, d], k_chunk/v_chunk [B, C, Hkv, d],
k/v of the sparse path [B, start_pos + C, Hkv, d].  A missing libpf.so is an
error (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpf.so")

PF_OK, PF_EINVAL, PF_EUNSUPPORTED, PF_ECUDA, PF_ETIMEOUT, PF_ERANGE = range(6)
PF_F16, PF_BF16, PF_F32 = range(3)
STATUS_NAMES = {0: "PF_OK", 1: "PF_EINVAL", 2: "PF_EUNSUPPORTED", 3: "PF_ECUDA", 4: "PF_ETIMEOUT",
                5: "PF_ERANGE"}

EXPORTS = ["pf_attn_dense", "pf_dense_workspace_bytes", "pf_dense_workspace_bytes_masked",
           "pf_attn_indexed", "pf_indexed_workspace_bytes",
           "pf_block_index", "pf_attn_sparse",
           "pf_sparse_query_sizes", "pf_convert_f16",
           "pf_stream_status", "pf_set_wait_timeout", "pf_set_debug_withhold", "pf_launch_count",
           "pf_last_error", "pf_version"]


class PFError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


I64x3 = ctypes.c_int64 * 3


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("C", ctypes.c_int32), ("in_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int), ("mask_dtype", ctypes.c_int), ("scale", ctypes.c_float),
                ("q_stride", I64x3), ("kh_stride", I64x3), ("kc_stride", I64x3),
                ("o_stride", I64x3), ("okv_stride", I64x3), ("mask_ld", ctypes.c_int64),
                ("v_f16", ctypes.c_int32)]


class Sel(ctypes.Structure):
    _fields_ = [("row_bits", ctypes.c_void_p), ("tile_list", ctypes.c_void_p),
                ("tile_cnt", ctypes.c_void_p), ("kbar", ctypes.c_void_p),
                ("capacity", ctypes.c_int32), ("pooled_blocks", ctypes.c_int32)]


class KeepRules(ctypes.Structure):
    """pf_keep_rules: sinks (tokens), local window (blocks), dense tail (rows), row_group
    (1 or 32), share_kv_group (0 or 1)."""
    _fields_ = [(n, ctypes.c_int32) for n in ("sink_tokens", "local_blocks", "dense_tail_rows",
                                              "row_group", "share_kv_group")]

    def __init__(self, sink_tokens=0, local_blocks=0, dense_tail_rows=0, row_group=1, share_kv_group=0):
        super().__init__(sink_tokens, local_blocks, dense_tail_rows, row_group, int(share_kv_group))


class SparseSizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("nblk", "nqt", "words", "row_bits_elems", "tile_list_elems",
                                              "tile_cnt_elems", "kbar_elems", "pooled_bytes")]


_lib = None


def load() -> ctypes.CDLL:
    """Load libpf.so (built by ``build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libpf.so not found at %s: run __graft_entry__.build() first" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    V, I32, I64, F, P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.POINTER
    lib.pf_attn_dense.argtypes = [P(Shape), V, V, V, V, V, V, I32, V, V, V, V, V, I64, V]
    lib.pf_dense_workspace_bytes.argtypes = [P(Shape), P(I64)]
    lib.pf_dense_workspace_bytes_masked.argtypes = [P(Shape), I32, P(I64)]
    lib.pf_attn_indexed.argtypes = [P(Shape), V, V, V, V, V, V, V, I32, I32, I32, V, V, V, V, V, I64, V]
    lib.pf_indexed_workspace_bytes.argtypes = [P(Shape), I32, P(I64)]
    lib.pf_block_index.argtypes = [P(Shape), V, V, I32, I32, F, P(KeepRules), P(Sel), V]
    lib.pf_attn_sparse.argtypes = [P(Shape), V, V, V, I32, I32, P(Sel), V, V, V, V]
    lib.pf_sparse_query_sizes.argtypes = [P(Shape), I32, I32, P(SparseSizes)]
    lib.pf_convert_f16.argtypes = [V, V, I64, V]
    lib.pf_stream_status.argtypes = [V]
    lib.pf_set_wait_timeout.argtypes = [I64]
    lib.pf_set_wait_timeout.restype = None
    lib.pf_set_debug_withhold.argtypes = [I32]
    lib.pf_set_debug_withhold.restype = None
    lib.pf_launch_count.argtypes = [I32]
    lib.pf_launch_count.restype = I64
    lib.pf_last_error.restype = ctypes.c_char_p
    lib.pf_version.restype = ctypes.c_char_p
    for name in ("pf_attn_dense", "pf_dense_workspace_bytes", "pf_dense_workspace_bytes_masked",
                 "pf_attn_indexed", "pf_indexed_workspace_bytes",
                 "pf_block_index", "pf_attn_sparse",
                 "pf_sparse_query_sizes", "pf_convert_f16", "pf_stream_status"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(rc: int):
    if rc != PF_OK:
        raise PFError(rc, load().pf_last_error().decode())


_DT = {torch.float16: PF_F16, torch.bfloat16: PF_BF16, torch.float32: PF_F32}


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError("unsupported dtype %s" % t.dtype)
    return _DT[t.dtype]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _bth(t: torch.Tensor):
    """(b, t, h) element strides of a [B, T, H, d] tensor with d contiguous."""
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("expected a [B, T, H, d] tensor with a contiguous last dim")
    return I64x3(t.stride(0), t.stride(1), t.stride(2))


def _same_layout(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Equal strides wherever the extent is above 1 (a size-1 dimension's stride is never
    used, and views of one-row slices keep their parent's)."""
    return a.shape == b.shape and all(sa == sb or n == 1 for sa, sb, n in zip(a.stride(), b.stride(), a.shape))


def _expect(t, shape, name, device):
    """Refuse a tensor whose extents differ from what the call will read or write: the C
    ABI takes bare pointers and cannot check them itself."""
    if t is None:
        raise ValueError("%s is required" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def _expect_selection(sel, z, B, C, Hq, Hkv, d, device):
    _expect(sel.row_bits, (B, Hq, C, z.words), "sel.row_bits", device)
    _expect(sel.tile_list, (B, Hq, z.nqt, z.nblk), "sel.tile_list", device)
    _expect(sel.tile_cnt, (B, Hq, z.nqt), "sel.tile_cnt", device)
    cap = sel.kbar.shape[3] if sel.kbar.dim() == 5 else -1
    if cap < z.nblk:
        raise ValueError("sel.kbar holds %d key blocks, this call needs %d" % (cap, z.nblk))
    _expect(sel.kbar, (2, B, Hkv, cap, d), "sel.kbar", device)
    if not sel.kbar.is_contiguous():
        raise ValueError("sel.kbar must be contiguous")


def _expect_lse(lse, B, Hq, C, device):
    if lse is None:
        return
    _expect(lse, (B, Hq, C), "lse", device)
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, Hq, C] tensor")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _v_flag(q, k, v, name="v") -> int:
    """k must have q's type; v either q's type or float16 (with bfloat16 q/k: the v_f16 mode,
    in which the kernels read v as it is instead of converting each tile)."""
    if k.dtype != q.dtype:
        raise TypeError("k has dtype %s, q has %s" % (k.dtype, q.dtype))
    if v.dtype == q.dtype:
        return 0
    if v.dtype == torch.float16 and q.dtype == torch.bfloat16:
        return 1
    raise TypeError("%s has dtype %s; expected %s or float16" % (name, v.dtype, q.dtype))


def make_shape(q, k_like, out_dtype, scale=0.0) -> Shape:
    B, C, Hq, d = q.shape
    sh = Shape()
    sh.B, sh.Hq, sh.Hkv, sh.d, sh.C = B, Hq, k_like.shape[2], d, C
    sh.in_dtype = _dtype(q)
    sh.out_dtype = _DT[out_dtype]
    sh.mask_dtype = PF_F32
    sh.scale = float(scale)
    sh.q_stride = _bth(q)
    return sh


_WORKSPACES = {}


def dense_workspace(q, stream=None, masked_start_pos=None) -> torch.Tensor:
    """The pf_attn_dense workspace (tail split; with masked_start_pos, also the packed bits of
    an explicit mask or of pf_attn_indexed's keep lists, whose workspace has the same size) for
    q, one per (device, stream) so that calls on different streams never share one."""
    lib = load()
    sh = Shape()
    sh.d = q.shape[-1]
    sh.C = q.shape[1]
    n = ctypes.c_int64(0)
    with torch.cuda.device(q.device):
        if masked_start_pos is None:
            _check(lib.pf_dense_workspace_bytes(ctypes.byref(sh), ctypes.byref(n)))
        else:
            _check(lib.pf_dense_workspace_bytes_masked(ctypes.byref(sh), int(masked_start_pos),
                                                       ctypes.byref(n)))
    key = (q.device, _stream(stream).value)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < int(n.value):
        ws = torch.empty((int(n.value),), dtype=torch.uint8, device=q.device)
        _WORKSPACES[key] = ws
    return ws


def attn_dense(q, k_hist, v_hist, k_chunk, v_chunk, start_pos, mask=None, out=None, out_k=None,
               out_v=None, out_dtype=torch.float32, scale=0.0, stream=None, workspace=True, lse=None):
    """Dense chunked prefill (pf_attn_dense); returns out [B, C, Hq, d].  workspace: True
    uses a cached per-(device, stream) buffer (tail split on), None runs every unit whole,
    or a caller-owned uint8 tensor of at least pf_dense_workspace_bytes.  lse: an optional
    fp32 [B, Hq, C] tensor that receives log sum_j exp(l_j) per row."""
    return _dense_call(q, k_hist, v_hist, k_chunk, v_chunk, start_pos, mask, None, out, out_k, out_v,
                       out_dtype, scale, stream, workspace, lse)


def attn_indexed(q, k_hist, v_hist, k_chunk, v_chunk, start_pos, keep_idx, keep_cnt, ratio, out=None,
                 out_k=None, out_v=None, out_dtype=torch.float32, scale=0.0, stream=None, workspace=True,
                 lse=None):
    """Index-driven attention (pf_attn_indexed): row i attends to the keys of its kept compressed
    blocks (keep_idx [C, S] int32, the first keep_cnt[i] entries of row i; block c covers keys
    ratio*c .. ratio*c + ratio - 1) plus the keys after its last complete block.  workspace:
    True (a cached buffer) or a caller-owned uint8 tensor of at least
    pf_indexed_workspace_bytes; the call needs one."""
    if workspace is None or workspace is False:
        raise ValueError("attn_indexed needs a workspace")
    C = q.shape[1] if q.dim() == 4 else -1
    if keep_idx.dim() != 2 or keep_idx.shape[0] != C or keep_idx.dtype != torch.int32 or \
            keep_idx.stride(1) != 1:
        raise ValueError("keep_idx must be an int32 [C, S] tensor with contiguous rows")
    _expect(keep_cnt, (C,), "keep_cnt", q.device)
    if keep_idx.device != q.device:
        raise ValueError("keep_idx is on %s, expected %s" % (keep_idx.device, q.device))
    if keep_cnt.dtype != torch.int32 or not keep_cnt.is_contiguous():
        raise ValueError("keep_cnt must be a contiguous int32 [C] tensor")
    keep = (keep_idx, keep_cnt, int(keep_idx.stride(0)), int(ratio))
    return _dense_call(q, k_hist, v_hist, k_chunk, v_chunk, start_pos, None, keep, out, out_k, out_v,
                       out_dtype, scale, stream, workspace, lse)


def _dense_call(q, k_hist, v_hist, k_chunk, v_chunk, start_pos, mask, keep, out, out_k, out_v, out_dtype,
                scale, stream, workspace, lse):
    lib = load()
    if q.dim() != 4:
        raise ValueError("q must be [B, C, Hq, d]")
    B, C, Hq, d = q.shape
    Hkv = k_chunk.shape[2] if k_chunk is not None and k_chunk.dim() == 4 else -1
    dev = q.device
    _expect(k_chunk, (B, C, Hkv, d), "k_chunk", dev)
    _expect(v_chunk, (B, C, Hkv, d), "v_chunk", dev)
    if start_pos > 0:
        _expect(k_hist, (B, start_pos, Hkv, d), "k_hist", dev)
        _expect(v_hist, (B, start_pos, Hkv, d), "v_hist", dev)
    if out is None:
        out = torch.empty((B, C, Hq, d), dtype=out_dtype, device=q.device)
    _expect(out, (B, C, Hq, d), "out", dev)
    if (out_k is None) != (out_v is None):
        raise ValueError("out_k and out_v go together")
    if out_k is not None:
        _expect(out_k, (B, Hkv, C, d), "out_k", dev)
        _expect(out_v, (B, Hkv, C, d), "out_v", dev)
    if mask is not None:
        _expect(mask, (C, start_pos + C), "mask", dev)
    _expect_lse(lse, B, Hq, C, dev)
    if workspace is True:
        workspace = dense_workspace(q, stream, None if mask is None and keep is None else start_pos)
    elif workspace is False:
        workspace = None
    if workspace is not None and workspace.device != dev:
        raise ValueError("workspace is on %s, expected %s" % (workspace.device, dev))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    sh = make_shape(q, k_chunk, out.dtype, scale)
    sh.v_f16 = _v_flag(q, k_chunk, v_chunk, "v_chunk")
    if start_pos > 0 and (k_hist.dtype != k_chunk.dtype or v_hist.dtype != v_chunk.dtype):
        raise TypeError("k_hist / v_hist must have the types of k_chunk / v_chunk")
    if out_k is not None and (out_k.dtype != k_chunk.dtype or out_v.dtype != v_chunk.dtype):
        raise TypeError("out_k / out_v must have the types of k_chunk / v_chunk")
    sh.kc_stride = _bth(k_chunk)
    if not _same_layout(v_chunk, k_chunk):
        raise ValueError("k_chunk and v_chunk must share strides")
    if start_pos > 0:
        sh.kh_stride = _bth(k_hist)
        if not _same_layout(v_hist, k_hist):
            raise ValueError("k_hist and v_hist must share strides")
    sh.o_stride = _bth(out)
    if out_k is not None:
        if not _same_layout(out_k, out_v) or out_k.stride(3) != 1:
            raise ValueError("out_k / out_v must share strides with a contiguous last dim")
        sh.okv_stride = I64x3(out_k.stride(0), out_k.stride(1), out_k.stride(2))  # (b, h, t)
    if mask is not None:
        if mask.dim() != 2 or mask.stride(1) != 1:
            raise ValueError("mask must be [C, start_pos + C] with contiguous rows")
        sh.mask_dtype = _dtype(mask)
        sh.mask_ld = mask.stride(0)
    kh = _ptr(k_hist if start_pos > 0 else None)
    vh = _ptr(v_hist if start_pos > 0 else None)
    if keep is None:
        _check(lib.pf_attn_dense(ctypes.byref(sh), _ptr(q), kh, vh, _ptr(k_chunk), _ptr(v_chunk),
                                 _ptr(mask), int(start_pos), _ptr(out), _ptr(lse), _ptr(out_k),
                                 _ptr(out_v), _ptr(workspace), int(ws_bytes), _stream(stream)))
    else:
        keep_idx, keep_cnt, stride, ratio = keep
        _check(lib.pf_attn_indexed(ctypes.byref(sh), _ptr(q), kh, vh, _ptr(k_chunk), _ptr(v_chunk),
                                   _ptr(keep_idx), _ptr(keep_cnt), stride, ratio, int(start_pos),
                                   _ptr(out), _ptr(lse), _ptr(out_k), _ptr(out_v), _ptr(workspace),
                                   int(ws_bytes), _stream(stream)))
    return out


def sparse_sizes(q, k, start_pos, block=128) -> SparseSizes:
    lib = load()
    sh = make_shape(q, k, torch.float32)
    z = SparseSizes()
    _check(lib.pf_sparse_query_sizes(ctypes.byref(sh), int(start_pos), int(block), ctypes.byref(z)))
    return z


@dataclasses.dataclass
class Selection:
    """Device buffers of a pf_sel: row_bits [B,Hq,C,W] int32 (bit pattern), tile_list
    [B,Hq,nqt,nblk], tile_cnt [B,Hq,nqt], kbar [2,B,Hkv,cap,d] fp32 (means, then the
    library's 16-bit hi/lo split of them; cap >= nblk blocks).  pooled_blocks: leading blocks
    that kbar (and the sparse workspace passed with this selection) already hold from an
    earlier chunk of the same prompt."""
    row_bits: torch.Tensor
    tile_list: torch.Tensor
    tile_cnt: torch.Tensor
    kbar: torch.Tensor
    pooled_blocks: int = 0

    @property
    def kbar_mean(self) -> torch.Tensor:
        return self.kbar[0]

    def c_struct(self) -> Sel:
        return Sel(self.row_bits.data_ptr(), self.tile_list.data_ptr(), self.tile_cnt.data_ptr(),
                   self.kbar.data_ptr(), int(self.kbar.shape[3]), int(self.pooled_blocks))


def alloc_kbar(q, k, max_keys, block=128) -> torch.Tensor:
    """A pooled-key buffer for a prompt of up to max_keys keys, [2, B, Hkv, ceil(max_keys /
    block), d] fp32: one buffer can serve every chunk of the prompt."""
    B, d, Hkv = q.shape[0], q.shape[3], k.shape[2]
    nblk = (int(max_keys) + block - 1) // block
    return torch.empty((2, B, Hkv, nblk, d), dtype=torch.float32, device=q.device)


def alloc_selection(q, k, start_pos, block=128, kbar=None, pooled_blocks=0) -> Selection:
    """Buffers for pf_block_index on this chunk.  kbar: a shared pooled-key buffer (alloc_kbar)
    that already holds the first pooled_blocks blocks of this prompt; None allocates one."""
    z = sparse_sizes(q, k, start_pos, block)
    B, C, Hq, d = q.shape
    Hkv = k.shape[2]
    dev = q.device
    if kbar is None:
        kbar = torch.empty((2, B, Hkv, z.nblk, d), dtype=torch.float32, device=dev)
    return Selection(torch.empty((B, Hq, C, z.words), dtype=torch.int32, device=dev),
                     torch.empty((B, Hq, z.nqt, z.nblk), dtype=torch.int32, device=dev),
                     torch.empty((B, Hq, z.nqt), dtype=torch.int32, device=dev),
                     kbar, int(pooled_blocks))


def block_index(q, k, start_pos, block=128, alpha=0.1, sel=None, scale=0.0, stream=None,
                rules: KeepRules = None) -> Selection:
    """Pooled block selection (pf_block_index); rules: optional KeepRules."""
    lib = load()
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, C, Hq, d] and k [B, start_pos + C, Hkv, d]")
    B, C, Hq, d = q.shape
    _expect(k, (B, start_pos + C, k.shape[2], d), "k", q.device)
    if sel is None:
        sel = alloc_selection(q, k, start_pos, block)
    _expect_selection(sel, sparse_sizes(q, k, start_pos, block), B, C, Hq, k.shape[2], d, q.device)
    sh = make_shape(q, k, torch.float32, scale)
    sh.kh_stride = _bth(k)
    cs = sel.c_struct()
    _check(lib.pf_block_index(ctypes.byref(sh), _ptr(q), _ptr(k), int(start_pos), int(block),
                              float(alpha), ctypes.byref(rules) if rules is not None else None,
                              ctypes.byref(cs), _stream(stream)))
    return sel


def alloc_pooled(q, k, start_pos, block=128, max_keys=None) -> torch.Tensor:
    """The pf_attn_sparse workspace; with max_keys, sized for a whole prompt of that many keys
    (to be shared by its chunks, together with a kbar from alloc_kbar(max_keys))."""
    if max_keys is not None:  # the sizes depend on the keys' count, not on k's contents
        start_pos = int(max_keys) - q.shape[1]
    z = sparse_sizes(q, k, start_pos, block)
    return torch.empty((z.pooled_bytes,), dtype=torch.uint8, device=q.device)


def attn_sparse(q, k, v, start_pos, sel: Selection, block=128, pooled=None, out=None,
                out_dtype=torch.float32, scale=0.0, stream=None, lse=None):
    """Block-sparse attention with pooled correction (pf_attn_sparse); returns out.  lse:
    an optional fp32 [B, Hq, C] tensor for the log of each row's denominator."""
    lib = load()
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, C, Hq, d] and k, v [B, start_pos + C, Hkv, d]")
    B, C, Hq, d = q.shape
    Hkv = k.shape[2]
    dev = q.device
    _expect(k, (B, start_pos + C, Hkv, d), "k", dev)
    _expect(v, (B, start_pos + C, Hkv, d), "v", dev)
    z = sparse_sizes(q, k, start_pos, block)
    _expect_selection(sel, z, B, C, Hq, Hkv, d, dev)
    cap = sel.kbar.shape[3]
    if cap != z.nblk:  # a workspace shared by a prompt's chunks is sized for its capacity
        pe = B * Hkv * cap * d
        z.pooled_bytes = (pe * 4 + 255) // 256 * 256 + 2 * ((pe * 2 + 255) // 256 * 256)
    if out is None:
        out = torch.empty((B, C, Hq, d), dtype=out_dtype, device=q.device)
    _expect(out, (B, C, Hq, d), "out", dev)
    _expect_lse(lse, B, Hq, C, dev)
    if pooled is None:
        pooled = alloc_pooled(q, k, start_pos, block)
    if pooled.device != dev or pooled.numel() * pooled.element_size() < z.pooled_bytes:
        raise ValueError("pooled must hold %d bytes on %s" % (z.pooled_bytes, dev))
    if not _same_layout(v, k):
        raise ValueError("k and v must share strides")
    sh = make_shape(q, k, out.dtype, scale)
    sh.v_f16 = _v_flag(q, k, v)
    sh.kh_stride = _bth(k)
    sh.o_stride = _bth(out)
    cs = sel.c_struct()
    _check(lib.pf_attn_sparse(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), int(start_pos), int(block),
                              ctypes.byref(cs), _ptr(pooled), _ptr(out), _ptr(lse), _stream(stream)))
    return out


def vbar_view(pooled: torch.Tensor, q, k, start_pos, block=128, capacity=None) -> torch.Tensor:
    """The fp32 block means of v at the head of the sparse workspace, [B, Hkv, cap, d] (cap =
    capacity, else this call's block count)."""
    z = sparse_sizes(q, k, start_pos, block)
    B, Hkv, d = q.shape[0], k.shape[2], q.shape[3]
    cap = z.nblk if capacity is None else int(capacity)
    return pooled[: B * Hkv * cap * d * 4].view(torch.float32).view(B, Hkv, cap, d)


def to_f16(x: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """bf16 -> fp16 copy of x (pf_convert_f16), for a v kept in fp16 (the v_f16 mode of the
    attention calls).  x and out contiguous, numel a multiple of 8; a value beyond fp16's
    range is reported by stream_status() as PF_ERANGE."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise TypeError("x must be a contiguous bfloat16 tensor")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    if out.dtype != torch.float16 or not out.is_contiguous() or out.numel() != x.numel() or out.device != x.device:
        raise ValueError("out must be a contiguous float16 tensor of x's size on x's device")
    _check(load().pf_convert_f16(_ptr(x), _ptr(out), int(x.numel()), _stream(stream)))
    return out


def stream_status(stream=None):
    _check(load().pf_stream_status(_stream(stream)))


def set_wait_timeout(cycles: int):
    load().pf_set_wait_timeout(int(cycles))


def set_debug_withhold(on: bool):
    load().pf_set_debug_withhold(1 if on else 0)


def launch_count(reset: bool = False) -> int:
    return int(load().pf_launch_count(1 if reset else 0))


def version() -> str:
    return load().pf_version().decode()
