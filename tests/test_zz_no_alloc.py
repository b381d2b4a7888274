"""pf_attn_sparse_static: block-sparse attention for callers that cannot allocate
device memory (a plug-in whose host framework owns all allocations, a serving
loop that must not call cudaMalloc).  Its scratch is a static buffer inside the
library; this checks it against pf_attn_sparse with a caller-allocated
workspace on two calls in a row, and that oversized problems are refused."""
import ctypes

import numpy as np
import pytest
import torch

import prefill_inputs as pi
from gpu_util import MAX_ABS, MEAN_ABS, dev, errors

pytestmark = pytest.mark.gpu

pfx = pytest.importorskip("long_context_prefill_chunked_gb300")
from long_context_prefill_chunked_gb300 import pf  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    lib = pfx.load()
    fn = lib.pf_attn_sparse_static
    V = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(pf.Shape), V, V, V, ctypes.c_int32, ctypes.c_int32,
                   ctypes.POINTER(pf.Sel), V, V, V]
    fn.restype = ctypes.c_int
    return lib


def call_static(lib, q, k, v, s, sel, out):
    sh = pf.make_shape(q, k, out.dtype)
    sh.kh_stride = pf._bth(k)
    sh.o_stride = pf._bth(out)
    cs = sel.c_struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pf_attn_sparse_static(ctypes.byref(sh), ctypes.c_void_p(q.data_ptr()),
                                     ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                     s, 128, ctypes.byref(cs), ctypes.c_void_p(out.data_ptr()), None,
                                     stream)


def test_static_scratch_matches_caller_workspace_two_calls(lib):
    big = pi.planted_workload("static-a", 31, 1, 8, 2, 128, 4096, 4096, "bf16")
    small = pi.planted_workload("static-b", 32, 1, 4, 2, 128, 1536, 1536, "bf16")
    for w, s in ((big, 0), (small, 512)):
        q = dev(w.q[:, s:], w.dtype)
        k, v = dev(w.k, w.dtype), dev(w.v, w.dtype)
        sel = pfx.block_index(q, k, s, 128, 0.1)
        ref = pfx.attn_sparse(q, k, v, s, sel)
        out = torch.full_like(ref, float("nan"))
        rc = call_static(lib, q, k, v, s, sel, out)
        assert rc == pf.PF_OK, lib.pf_last_error().decode()
        pfx.stream_status()
        mx, mean = errors(out, ref.double().cpu().numpy())
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)


def test_static_scratch_refuses_oversized_problems(lib):
    sh = pf.Shape()
    sh.B, sh.Hq, sh.Hkv, sh.d, sh.C = 2, 32, 8, 128, 2048 * 128   # 32 MiB of scratch
    sh.in_dtype, sh.out_dtype, sh.mask_dtype = pf.PF_BF16, pf.PF_F32, pf.PF_F32
    fake = ctypes.c_void_p(0x100000)
    sel = pf.Sel(0x100000, 0x100000, 0x100000, 0x100000)
    rc = lib.pf_attn_sparse_static(ctypes.byref(sh), fake, fake, fake, 0, 128, ctypes.byref(sel), fake, None,
                                   None)
    assert rc == pf.PF_EUNSUPPORTED
    assert b"static buffer" in lib.pf_last_error()


@pytest.mark.parametrize("field,value,start", [("C", 0, 0), ("B", -1, 0), ("Hkv", 0, 0), ("d", -128, 0),
                                               ("C", 4096, -128)])
def test_static_scratch_refuses_invalid_shapes(lib, field, value, start):
    """An invalid shape is PF_EINVAL (as pf_attn_sparse gives), not a scratch-size refusal."""
    sh = pf.Shape()
    sh.B, sh.Hq, sh.Hkv, sh.d, sh.C = 1, 8, 2, 128, 4096
    sh.in_dtype, sh.out_dtype, sh.mask_dtype = pf.PF_BF16, pf.PF_F32, pf.PF_F32
    setattr(sh, field, value)
    fake = ctypes.c_void_p(0x100000)
    sel = pf.Sel(0x100000, 0x100000, 0x100000, 0x100000)
    rc = lib.pf_attn_sparse_static(ctypes.byref(sh), fake, fake, fake, start, 128, ctypes.byref(sel), fake,
                                   None, None)
    assert rc == pf.PF_EINVAL, (rc, lib.pf_last_error())
    assert b"static buffer" not in lib.pf_last_error()
