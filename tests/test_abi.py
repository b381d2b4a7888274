"""The C ABI without a GPU: the library loads, exports what include/pf.h declares,
and refuses bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import long_context_prefill_chunked_gb300 as pfx
from long_context_prefill_chunked_gb300 import pf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pf.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return pfx.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:pf_status|void|int64_t|const char\*)\s+(pf_\w+)\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "pf_attn_dense" in names and "pf_block_index" in names and "pf_attn_sparse" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(pf.EXPORTS) <= set(names)


def test_version(lib):
    assert "sm_103a" in pfx.version()


def shape(**kw):
    sh = pf.Shape()
    sh.B, sh.Hq, sh.Hkv, sh.d, sh.C = 1, 4, 2, 128, 256
    sh.in_dtype, sh.out_dtype, sh.mask_dtype = pf.PF_BF16, pf.PF_F32, pf.PF_F32
    for k, v in kw.items():
        setattr(sh, k, v)
    return sh


FAKE = ctypes.c_void_p(0x100000)      # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x100008)


def dense(lib, sh, q=FAKE, kh=None, vh=None, kc=FAKE, vc=FAKE, mask=None, s=0, out=FAKE, ok=None, ov=None,
          ws=None, ws_bytes=0):
    return lib.pf_attn_dense(ctypes.byref(sh) if sh is not None else None, q, kh, vh, kc, vc, mask, s,
                             out, None, ok, ov, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), pf.PF_EUNSUPPORTED),
    (dict(d=512), pf.PF_EUNSUPPORTED),
    (dict(Hq=6, Hkv=4), pf.PF_EINVAL),
    (dict(C=0), pf.PF_EINVAL),
    (dict(in_dtype=pf.PF_F32), pf.PF_EUNSUPPORTED),
    (dict(scale=-1.0), pf.PF_EINVAL),
    (dict(v_f16=2), pf.PF_EINVAL),
])
def test_dense_rejects_bad_shapes(lib, kw, code):
    assert dense(lib, shape(**kw)) == code
    assert lib.pf_last_error()


def test_dense_rejects_bad_arguments(lib):
    assert dense(lib, None) == pf.PF_EINVAL
    assert dense(lib, shape(), q=None) == pf.PF_EINVAL
    assert dense(lib, shape(), s=100, kh=FAKE, vh=FAKE) == pf.PF_EUNSUPPORTED   # start_pos % 128
    assert dense(lib, shape(), s=128) == pf.PF_EINVAL                           # history missing
    assert dense(lib, shape(), s=-128) == pf.PF_EINVAL
    assert dense(lib, shape(), q=MISALIGNED) == pf.PF_EINVAL
    assert dense(lib, shape(), ok=FAKE) == pf.PF_EINVAL                         # out_v missing
    assert dense(lib, shape(mask_dtype=pf.PF_BF16), mask=FAKE) == pf.PF_EUNSUPPORTED
    bad = shape()
    bad.q_stride = pf.I64x3(256 * 4 * 128, 4 * 128, 60)                          # 120-byte head stride
    assert dense(lib, bad) == pf.PF_EINVAL


def indexed(lib, sh, keep_idx=FAKE, keep_cnt=FAKE, stride=16, ratio=4, s=0, ws=FAKE, ws_bytes=1 << 30):
    return lib.pf_attn_indexed(ctypes.byref(sh), FAKE, None, None, FAKE, FAKE, keep_idx, keep_cnt, stride,
                               ratio, s, FAKE, None, None, None, ws, ws_bytes, None)


def test_indexed_rejects_bad_arguments(lib):
    sh = shape()
    assert indexed(lib, sh, ratio=0) == pf.PF_EINVAL
    assert indexed(lib, sh, ratio=129) == pf.PF_EINVAL
    assert indexed(lib, sh, keep_cnt=None) == pf.PF_EINVAL
    assert indexed(lib, sh, keep_idx=None) == pf.PF_EINVAL                  # entries but no list
    assert indexed(lib, sh, stride=-1) == pf.PF_EINVAL
    assert indexed(lib, sh, keep_idx=ctypes.c_void_p(0x100002)) == pf.PF_EINVAL
    assert indexed(lib, sh, ws=None) == pf.PF_EINVAL                        # the bits need a workspace
    assert indexed(lib, shape(C=(1 << 20) + 128)) == pf.PF_EUNSUPPORTED     # past 2^20 keys
    assert b"1048576" in lib.pf_last_error()


def test_sparse_rejects_bad_arguments(lib):
    sel = pf.Sel(0x100000, 0x100000, 0x100000, 0x100000)
    sh = shape()
    assert lib.pf_block_index(ctypes.byref(sh), FAKE, FAKE, 0, 64, 0.1, None, ctypes.byref(sel), None) == pf.PF_EUNSUPPORTED
    assert lib.pf_block_index(ctypes.byref(sh), FAKE, FAKE, 0, 128, 1.5, None, ctypes.byref(sel), None) == pf.PF_EUNSUPPORTED
    assert lib.pf_block_index(ctypes.byref(sh), FAKE, FAKE, 0, 128, -0.1, None, ctypes.byref(sel), None) == pf.PF_EUNSUPPORTED
    assert lib.pf_block_index(ctypes.byref(sh), None, FAKE, 0, 128, 0.1, None, ctypes.byref(sel), None) == pf.PF_EINVAL
    bad_group = pf.KeepRules(row_group=16)
    assert lib.pf_block_index(ctypes.byref(sh), FAKE, FAKE, 0, 128, 0.1, ctypes.byref(bad_group),
                              ctypes.byref(sel), None) == pf.PF_EUNSUPPORTED
    bad_count = pf.KeepRules(sink_tokens=-1)
    assert lib.pf_block_index(ctypes.byref(sh), FAKE, FAKE, 0, 128, 0.1, ctypes.byref(bad_count),
                              ctypes.byref(sel), None) == pf.PF_EINVAL
    assert lib.pf_attn_sparse(ctypes.byref(sh), FAKE, FAKE, FAKE, 0, 128, ctypes.byref(sel), None, FAKE, None, None) == pf.PF_EINVAL
    long = shape(C=300000)
    assert lib.pf_attn_sparse(ctypes.byref(long), FAKE, FAKE, FAKE, 0, 128, ctypes.byref(sel), FAKE, FAKE, None, None) == pf.PF_EUNSUPPORTED


def test_sparse_pooled_reuse_arguments(lib):
    """capacity below the call's block count, or pooled_blocks beyond the whole history blocks
    (or negative), is PF_EINVAL for both sparse calls, before anything is launched."""
    sh = shape(C=256)                                           # start_pos 512: nblk 6, 4 history blocks
    for cap, pooled in ((5, 0), (-1, 0), (8, 5), (8, -1)):
        sel = pf.Sel(0x100000, 0x100000, 0x100000, 0x100000, cap, pooled)
        assert lib.pf_block_index(ctypes.byref(sh), FAKE, FAKE, 512, 128, 0.1, None, ctypes.byref(sel),
                                  None) == pf.PF_EINVAL, (cap, pooled)
        assert lib.pf_attn_sparse(ctypes.byref(sh), FAKE, FAKE, FAKE, 512, 128, ctypes.byref(sel), FAKE, FAKE,
                                  None, None) == pf.PF_EINVAL, (cap, pooled)
    big = pf.Sel(0x100000, 0x100000, 0x100000, 0x100000, 4096, 0)
    assert lib.pf_block_index(ctypes.byref(sh), FAKE, FAKE, 512, 128, 0.1, None, ctypes.byref(big),
                              None) == pf.PF_EUNSUPPORTED


def test_sparse_sizes(lib):
    sh = shape(C=4096, Hq=32, Hkv=8)
    z = pf.SparseSizes()
    assert lib.pf_sparse_query_sizes(ctypes.byref(sh), 8192, 128, ctypes.byref(z)) == pf.PF_OK
    assert (z.nblk, z.nqt, z.words) == (96, 32, 3)
    assert z.row_bits_elems == 32 * 4096 * 3
    assert z.tile_list_elems == 32 * 32 * 96
    assert z.kbar_elems == 2 * 8 * 96 * 128
    assert z.pooled_bytes >= z.kbar_elems // 2 * (4 + 2 + 2)


def test_header_cites_the_pages():
    text = open(HEADER).read()
    for page in ("ANE Prefill Research", "Porting FlashPrefill V2 to Apple silicon"):
        assert page in text


def test_binding_refuses_mismatched_extents(lib):
    """The C ABI takes bare pointers; the binding must refuse a buffer whose extents differ from
    what the call reads or writes (these raise before any library call, so CPU tensors do)."""
    import torch
    B, C, Hq, Hkv, d, s = 1, 256, 4, 2, 128, 128
    bf = torch.bfloat16
    q = torch.zeros((B, C, Hq, d), dtype=bf)
    kc = torch.zeros((B, C, Hkv, d), dtype=bf)
    kh = torch.zeros((B, s, Hkv, d), dtype=bf)
    with pytest.raises(ValueError, match="out"):            # output with the wrong row count
        pf.attn_dense(q, kh, kh, kc, kc, s, out=torch.zeros((B, 4 * C, Hq, d)))
    with pytest.raises(ValueError, match="k_chunk"):        # chunk keys shorter than the queries
        pf.attn_dense(q, kh, kh, kc[:, :128], kc[:, :128], s)
    with pytest.raises(ValueError, match="k_hist"):         # history shorter than start_pos
        pf.attn_dense(q, kh[:, :64], kh[:, :64], kc, kc, s)
    with pytest.raises(ValueError, match="out_k"):          # cache slice of the wrong length
        pf.attn_dense(q, kh, kh, kc, kc, s, out=torch.zeros((B, C, Hq, d)),
                      out_k=torch.zeros((B, Hkv, C // 2, d), dtype=bf),
                      out_v=torch.zeros((B, Hkv, C // 2, d), dtype=bf))
    with pytest.raises(ValueError, match="mask"):
        pf.attn_dense(q, kh, kh, kc, kc, s, out=torch.zeros((B, C, Hq, d)),
                      mask=torch.zeros((C, C)))
    k_all = torch.zeros((B, s + C, Hkv, d), dtype=bf)
    with pytest.raises(ValueError, match="k"):
        pf.block_index(q, k_all[:, :C], s)


def test_binding_refuses_bad_keep_lists(lib):
    """attn_indexed: the keep lists must be int32 [C, S] with contiguous rows and keep_cnt an
    int32 [C] tensor, and a workspace is required (all raise before any library call)."""
    import torch
    B, C, Hq, Hkv, d, s = 1, 256, 4, 2, 128, 128
    bf = torch.bfloat16
    q = torch.zeros((B, C, Hq, d), dtype=bf)
    kc = torch.zeros((B, C, Hkv, d), dtype=bf)
    kh = torch.zeros((B, s, Hkv, d), dtype=bf)
    idx = torch.zeros((C, 8), dtype=torch.int32)
    cnt = torch.zeros((C,), dtype=torch.int32)
    with pytest.raises(ValueError, match="keep_idx"):
        pf.attn_indexed(q, kh, kh, kc, kc, s, idx.long(), cnt, 4)
    with pytest.raises(ValueError, match="keep_idx"):
        pf.attn_indexed(q, kh, kh, kc, kc, s, idx[:128], cnt, 4)
    with pytest.raises(ValueError, match="keep_idx"):
        pf.attn_indexed(q, kh, kh, kc, kc, s, idx.t().contiguous().t(), cnt, 4)
    with pytest.raises(ValueError, match="keep_cnt"):
        pf.attn_indexed(q, kh, kh, kc, kc, s, idx, cnt[:100], 4)
    with pytest.raises(ValueError, match="keep_cnt"):
        pf.attn_indexed(q, kh, kh, kc, kc, s, idx, cnt.long(), 4)
    with pytest.raises(ValueError, match="workspace"):
        pf.attn_indexed(q, kh, kh, kc, kc, s, idx, cnt, 4, workspace=None)


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "pf.h"

int main(void) {
  pf_shape sh;
  memset(&sh, 0, sizeof(sh));
  sh.B = 1; sh.Hq = 4; sh.Hkv = 2; sh.d = 128; sh.C = 256;
  sh.in_dtype = PF_BF16; sh.out_dtype = PF_F32; sh.mask_dtype = PF_F32;
  void* fake = (void*)0x100000;
  int32_t cnt = 0;
  if (strstr(pf_version(), "sm_103a") == NULL) return 1;
  if (pf_attn_dense(NULL, fake, NULL, NULL, fake, fake, NULL, 0, fake, NULL, NULL, NULL, NULL, 0, NULL)
      != PF_EINVAL) return 2;
  if (pf_attn_indexed(&sh, fake, NULL, NULL, fake, fake, (const int32_t*)fake, &cnt, 8, 0, 0, fake, NULL,
                      NULL, NULL, fake, 1, NULL) != PF_EINVAL) return 3;
  if (pf_last_error()[0] == '\0') return 4;
  printf("ok\n");
  return 0;
}
"""


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/pf.h compiles as C99 with warnings as errors, and a C program linked against
    libpf.so reaches the validation paths (no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    libdir = os.path.dirname(pf.LIB_PATH)
    exe = tmp_path / "caller"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lpf", "-Wl,-rpath," + libdir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)


def test_package_exports_every_binding_function():
    """Every public function of the binding module is reachable from the package."""
    import inspect
    import long_context_prefill_chunked_gb300 as pkg
    from long_context_prefill_chunked_gb300 import pf as mod
    public = [n for n, f in vars(mod).items() if inspect.isfunction(f) and not n.startswith("_")
              and f.__module__ == mod.__name__ and n != "make_shape"]
    missing = [n for n in public if not hasattr(pkg, n)]
    assert not missing, missing


def test_binding_v_type_and_layout_rules():
    """The binding's v type rule (v in q's type, or fp16 with bf16 q/k: the v_f16 flag) and its
    stride comparison (size-1 dimensions ignored: a one-row batch view keeps its parent's
    batch stride)."""
    import torch
    bq = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    assert pf._v_flag(bq, bq, bq) == 0
    assert pf._v_flag(bq, bq, bq.half()) == 1
    hq = bq.half()
    assert pf._v_flag(hq, hq, hq) == 0
    with pytest.raises(TypeError):
        pf._v_flag(bq, bq, bq.float())
    with pytest.raises(TypeError):
        pf._v_flag(bq, bq.half(), bq)
    with pytest.raises(TypeError):
        pf._v_flag(hq, hq, bq)
    big = torch.zeros(1, 12, 2, 64, dtype=torch.bfloat16)
    view = big[:, 4:8]                  # batch stride 12*2*64, the fresh tensor's is 4*2*64
    fresh = torch.zeros(1, 4, 2, 64, dtype=torch.float16)
    assert view.stride(0) != fresh.stride(0) and pf._same_layout(view, fresh)
    two = torch.zeros(2, 12, 2, 64, dtype=torch.bfloat16)[:, 4:8]
    assert not pf._same_layout(two, torch.zeros(2, 4, 2, 64, dtype=torch.float16))
    assert not pf._same_layout(fresh, fresh.transpose(1, 2))
