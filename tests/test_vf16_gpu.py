"""v kept in fp16 (the v_f16 mode): bf16 q/k with an fp16 v that pf_convert_f16 produced.

The attention kernels compute P * V in fp16 and otherwise convert each bf16 v tile in every CTA
that loads it; with v already in fp16 they read it as it is.  The conversion is the same
(bf16 -> fp32 exactly, rounded to nearest fp16), so the dense and index-driven outputs must be
bit-identical to the bf16-v path; the block-sparse path rounds its pooled means of v straight
to fp16 instead of through bf16, so it is compared with the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import prefill_inputs as pi
from gpu_util import MAX_ABS, MEAN_ABS, assert_close, dev

pytestmark = pytest.mark.gpu

pfx = pytest.importorskip("long_context_prefill_chunked_gb300")
from long_context_prefill_chunked_gb300 import pf  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    pfx.set_wait_timeout(400_000_000)
    yield
    pfx.stream_status()


def bf16_of(x: np.ndarray) -> torch.Tensor:
    """float32 values -> their bf16 bit patterns (round to nearest even) as a CUDA tensor."""
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).cuda()


def test_to_f16_exact_against_numpy():
    """Every bf16 value, small ones included, converts as numpy's float32 -> float16 does
    (round to nearest even); 65280, the largest bf16 value below fp16's limit 65504, passes."""
    g = np.random.default_rng(61)
    x = np.concatenate([[65280.0, -65280.0, 0.0, -0.0, 2.0 ** -24, 3e-8, 2.0 ** -25, 1.5 * 2.0 ** -24],
                        g.standard_normal(8192), g.standard_normal(1024) * 1e-6, g.standard_normal(1024) * 1e-9,
                        g.uniform(-65000, 65000, 1024)])
    assert len(x) % 8 == 0
    xb = bf16_of(x)
    got = pfx.to_f16(xb)
    pfx.stream_status()
    want = xb.float().cpu().numpy().astype(np.float16)
    assert np.array_equal(got.cpu().numpy().view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("bad", [70000.0, float("inf"), float("nan")])
def test_to_f16_out_of_range_reports_erange(bad):
    x = np.zeros(64, dtype=np.float32)
    x[17] = bad
    pfx.to_f16(bf16_of(x))
    with pytest.raises(pfx.PFError) as e:
        pfx.stream_status()
    assert e.value.status == pf.PF_ERANGE
    pfx.stream_status()  # cleared


def test_to_f16_refuses_misuse():
    with pytest.raises(TypeError):
        pfx.to_f16(torch.zeros(64, dtype=torch.float16, device="cuda"))
    lib = pfx.load()
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(64, dtype=torch.float16, device="cuda")
    assert lib.pf_convert_f16(pf._ptr(x), pf._ptr(y), 60, None) == pf.PF_EINVAL  # not a multiple of 8


@pytest.fixture(scope="module")
def w():
    return pi.normal_workload("vf16", 62, 1, 8, 2, 128, 1024, 300, "bf16")


def views(w, s, C):
    q = dev(w.q[:, s:s + C], "bf16")
    kh, kc = dev(w.k[:, :s], "bf16"), dev(w.k[:, s:s + C], "bf16")
    vh, vc = dev(w.v[:, :s], "bf16"), dev(w.v[:, s:s + C], "bf16")
    return q, kh, vh, kc, vc


@pytest.mark.parametrize("s", [0, 512])
@pytest.mark.parametrize("masked", [False, True])
def test_dense_fp16_v_bit_identical(w, s, masked):
    """Causal (with the tail-split workspace) and explicit-mask chunks over a history, K/V cache
    re-emitted: the fp16-v call equals the bf16-v call bit for bit, and out_v holds the fp16 v."""
    C = 300
    q, kh, vh, kc, vc = views(w, s, C)
    mask = None
    if masked:
        g = np.random.default_rng(63)
        m = np.where(g.random((C, s + C)) < 0.3, -30000.0, 0.0).astype(np.float32)
        m[:, 0] = 0.0
        mask = torch.from_numpy(m).cuda()
    ok16 = torch.empty((1, 2, C, 128), dtype=torch.bfloat16, device="cuda")
    ov16 = torch.empty((1, 2, C, 128), dtype=torch.float16, device="cuda")
    okb, ovb = torch.empty_like(ok16), torch.empty_like(ok16)
    ref = pfx.attn_dense(q, kh, vh, kc, vc, s, mask=mask, out_k=okb, out_v=ovb)
    vh16 = pfx.to_f16(vh.contiguous()) if s > 0 else vh[:, :0].half()
    vc16 = pfx.to_f16(vc.contiguous())
    out = pfx.attn_dense(q, kh, vh16, kc, vc16, s, mask=mask, out_k=ok16, out_v=ov16)
    pfx.stream_status()
    assert torch.equal(out, ref)
    assert torch.equal(ok16, okb)
    assert torch.equal(ov16, vc16.transpose(1, 2))
    want = oracle.dense(*(w.f64(x) for x in w.chunk_views(s)), s,
                        mask=None if mask is None else mask.cpu().numpy().astype(np.float64))[:, :C]
    assert_close(out, want, "fp16 v s=%d masked=%s" % (s, masked))


def test_indexed_fp16_v_bit_identical(w):
    s, C, ratio = 512, 300, 4
    q, kh, vh, kc, vc = views(w, s, C)
    g = np.random.default_rng(64)
    kept = [np.sort(g.choice((s + i + 1) // ratio, size=min((s + i + 1) // ratio, 30), replace=False))
            for i in range(C)]
    idx = np.full((C, 30), -1, dtype=np.int32)
    cnt = np.zeros(C, dtype=np.int32)
    for i, k in enumerate(kept):
        idx[i, :len(k)] = k
        cnt[i] = len(k)
    ti, tc = torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()
    ref = pfx.attn_indexed(q, kh, vh, kc, vc, s, ti, tc, ratio)
    out = pfx.attn_indexed(q, kh, pfx.to_f16(vh.contiguous()), kc, pfx.to_f16(vc.contiguous()), s, ti, tc, ratio)
    pfx.stream_status()
    assert torch.equal(out, ref)


def test_dense_fp16_v_head_dim_256():
    """Head dim 256 (64-key tiles, one head per CTA): fp16 v equals the bf16-v call bit for bit."""
    w = pi.normal_workload("vf16-d256", 66, 1, 4, 2, 256, 768, 437, "bf16")
    s, C = 256, 437
    q = dev(w.q[:, s:s + C], "bf16")
    kh, kc = dev(w.k[:, :s], "bf16"), dev(w.k[:, s:s + C], "bf16")
    vh, vc = dev(w.v[:, :s], "bf16"), dev(w.v[:, s:s + C], "bf16")
    ref = pfx.attn_dense(q, kh, vh, kc, vc, s)
    out = pfx.attn_dense(q, kh, pfx.to_f16(vh.contiguous()), kc, pfx.to_f16(vc.contiguous()), s)
    pfx.stream_status()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("s,C,d", [(0, 1536, 128), (512, 1024, 128), (512, 1024, 256)])
def test_sparse_fp16_v_matches_oracle(s, C, d):
    w = pi.planted_workload("vf16-sparse", 65, 1, 4, 2, d, 1536, 1536, "bf16")
    C = min(C, w.N - s)
    q = dev(w.q[:, s:s + C], "bf16")
    k = dev(w.k[:, :s + C], "bf16")
    v16 = pfx.to_f16(dev(w.v[:, :s + C], "bf16").contiguous())
    sel = pfx.block_index(q, k, s, 128, 0.1)
    out = pfx.attn_sparse(q, k, v16, s, sel)
    pfx.stream_status()
    nblk = (s + C + 127) // 128
    words = sel.row_bits.cpu().numpy().view(np.uint32)
    bits = np.unpackbits(words.view(np.uint8).reshape(*words.shape, 4), axis=-1, bitorder="little")
    gk = np.transpose(bits.reshape(*words.shape[:3], -1)[..., :nblk].astype(bool), (0, 2, 1, 3))
    ref, _, _ = oracle.sparse_for_selection(w.f64(w.q[:, s:s + C]), w.f64(w.k[:, :s + C]),
                                            w.f64(w.v[:, :s + C]), s, 128, 0.1, gk)
    e = np.abs(out.cpu().double().numpy() - ref)
    assert e.max() <= MAX_ABS and e.mean() <= MEAN_ABS, (e.max(), e.mean())


def test_v_dtype_checks(w):
    q, kh, vh, kc, vc = views(w, 512, 300)
    with pytest.raises(TypeError):  # fp32 v
        pfx.attn_dense(q, kh, vh.float(), kc, vc.float(), 512)
    with pytest.raises(TypeError):  # history and chunk of different types
        pfx.attn_dense(q, kh, vh, kc, pfx.to_f16(vc.contiguous()), 512)
