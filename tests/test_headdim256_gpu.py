"""Head dim 256 through the C ABI against the float64 oracle: dense causal and explicit-mask
chunked prefill (values and packed bits, with and without the tail split), index-driven
attention over keep lists, and block-sparse prefill with the pooled correction.  At this head
dim the kernels run 64-key tiles and one query head per CTA; chunks are ragged (not a multiple
of 128 rows) and start over a history."""
import numpy as np
import pytest
import torch

import oracle
import prefill_inputs as pi
from gpu_util import MAX_ABS, MEAN_ABS, assert_close, dev, errors

pytestmark = pytest.mark.gpu

pfx = pytest.importorskip("long_context_prefill_chunked_gb300")

D = 256
LSE_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    pfx.set_wait_timeout(400_000_000)
    yield
    pfx.stream_status()


@pytest.fixture(scope="module")
def w():
    # 4 query heads over 2 KV heads, 1024 tokens; chunks below are ragged
    return pi.normal_workload("d256", 41, 1, 4, 2, D, 1024, 512, "bf16")


def chunk(w, s, C):
    q, kh, vh = w.q[:, s:s + C], w.k[:, :s], w.v[:, :s]
    kc, vc = w.k[:, s:s + C], w.v[:, s:s + C]
    return (q, kh, vh, kc, vc)


@pytest.mark.parametrize("s,C", [(0, 300), (256, 437), (512, 512)])
@pytest.mark.parametrize("workspace", [True, None])
def test_dense_causal(w, s, C, workspace):
    parts = chunk(w, s, C)
    lse = torch.empty((1, w.Hq, C), dtype=torch.float32, device="cuda")
    out = pfx.attn_dense(*(dev(x, w.dtype) for x in parts), s, lse=lse, workspace=workspace)
    pfx.stream_status()
    ref, rlse = oracle.dense(*(w.f64(x) for x in parts), s, with_lse=True)
    assert_close(out, ref, "d256 causal s=%d C=%d" % (s, C))
    got = lse.cpu().double().numpy().transpose(0, 2, 1)
    assert np.max(np.abs(got - rlse)) <= LSE_TOL


@pytest.mark.parametrize("kind", ["values", "binary"])
def test_dense_explicit_mask(w, kind):
    """A non-binary mask runs the value path; a 0 / -30000 mask with the masked workspace runs
    the packed-bits path that skips key tiles no row keeps."""
    s, C = 256, 437
    parts = chunk(w, s, C)
    g = np.random.default_rng(43)
    if kind == "values":
        mask = g.uniform(-3.0, 1.0, size=(C, s + C)).astype(np.float32)
        ws = True
    else:
        mask = np.where(g.random((C, s + C)) < 0.4, -30000.0, 0.0).astype(np.float32)
        mask[:, 64:192] = -30000.0                                  # two dropped 64-key tiles
        mask[:, 0] = 0.0                                            # every row keeps a key
        ws = pfx.dense_workspace(dev(parts[0], w.dtype), masked_start_pos=s)
    out = pfx.attn_dense(*(dev(x, w.dtype) for x in parts), s, mask=torch.from_numpy(mask).cuda(),
                         workspace=ws)
    pfx.stream_status()
    ref = oracle.dense(*(w.f64(x) for x in parts), s, mask=mask.astype(np.float64))
    assert_close(out, ref, "d256 mask " + kind)


def test_indexed_keep_lists(w):
    """Keep lists of compressed blocks (ratio 4) over a 512-token history."""
    s, C, ratio = 512, 300, 4
    parts = chunk(w, s, C)
    g = np.random.default_rng(44)
    kept = []
    for i in range(C):
        nc = (s + i + 1) // ratio
        kept.append(np.sort(g.choice(nc, size=min(nc, 40), replace=False)).astype(np.int32))
    stride = max(len(k) for k in kept)
    idx = np.full((C, stride), -1, dtype=np.int32)
    cnt = np.zeros(C, dtype=np.int32)
    for i, k in enumerate(kept):
        idx[i, :len(k)] = k
        cnt[i] = len(k)
    out = pfx.attn_indexed(*(dev(x, w.dtype) for x in parts), s, torch.from_numpy(idx).cuda(),
                           torch.from_numpy(cnt).cuda(), ratio)
    pfx.stream_status()
    ref = oracle.dense_indexed(*(w.f64(x) for x in parts), s, kept, ratio)
    assert_close(out, ref, "d256 indexed")


@pytest.fixture(scope="module")
def planted():
    return pi.planted_workload("d256-sparse", 45, 1, 4, 2, D, 1536, 1536, "bf16")


@pytest.mark.parametrize("s,C", [(0, 1536), (512, 1024), (768, 700)])
def test_sparse_selection_and_output(planted, s, C):
    w = planted
    C = min(C, w.N - s)
    q = dev(w.q[:, s:s + C], w.dtype)
    k = dev(w.k[:, :s + C], w.dtype)
    v = dev(w.v[:, :s + C], w.dtype)
    sel = pfx.block_index(q, k, s, 128, 0.1)
    out = pfx.attn_sparse(q, k, v, s, sel)
    pfx.stream_status()
    nblk = (s + C + 127) // 128
    words = sel.row_bits.cpu().numpy().view(np.uint32)
    bits = np.unpackbits(words.view(np.uint8).reshape(*words.shape, 4), axis=-1, bitorder="little")
    gk = np.transpose(bits.reshape(*words.shape[:3], -1)[..., :nblk].astype(bool), (0, 2, 1, 3))
    ref, osel, _ = oracle.sparse_for_selection(w.f64(w.q[:, s:s + C]), w.f64(w.k[:, :s + C]),
                                               w.f64(w.v[:, :s + C]), s, 128, 0.1, gk)
    ok = ~osel.near
    assert np.array_equal(gk[ok], osel.kept[ok])
    e = np.abs(out.cpu().double().numpy() - ref)
    assert e.max() <= MAX_ABS and e.mean() <= MEAN_ABS, (e.max(), e.mean())
    assert oracle.skip_share(osel) > 0.3


def test_sparse_alpha_zero_equals_dense(planted):
    w = planted
    q, k, v = dev(w.q, w.dtype), dev(w.k, w.dtype), dev(w.v, w.dtype)
    sel = pfx.block_index(q, k, 0, 128, 0.0)
    out = pfx.attn_sparse(q, k, v, 0, sel)
    dense = pfx.attn_dense(q, k[:, :0], v[:, :0], k, v, 0)
    pfx.stream_status()
    mx, _ = errors(out, dense.double().cpu().numpy())
    assert mx <= 2e-3
