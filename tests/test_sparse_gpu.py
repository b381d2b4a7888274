"""Block-sparse prefill: selection bit-exact (outside the 1e-4 threshold band) and
outputs within tolerance of the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import prefill_inputs as pi
from gpu_util import MAX_ABS, assert_close, dev, errors, sample_rows
from long_context_prefill_chunked_gb300 import pf

pytestmark = pytest.mark.gpu

pfx = pytest.importorskip("long_context_prefill_chunked_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    pfx.set_wait_timeout(400_000_000)
    yield
    pfx.stream_status()


def gpu_bits_to_kept(row_bits: torch.Tensor, nblk: int) -> np.ndarray:
    """row_bits [B, Hq, C, W] -> bool [B, C, Hq, nblk]."""
    w = row_bits.cpu().numpy().view(np.uint32)
    bits = np.unpackbits(w.view(np.uint8).reshape(*w.shape, 4), axis=-1, bitorder="little")
    bits = bits.reshape(*w.shape[:3], -1)[..., :nblk].astype(bool)
    return np.transpose(bits, (0, 2, 1, 3))


def check_selection(sel, osel, rows, n_qt_check=None):
    """Row bits equal on every non-near row; tile lists equal unless a near row contributes."""
    nblk = osel.kept.shape[-1]
    gk = gpu_bits_to_kept(sel.row_bits, nblk)[:, rows]                   # [B, R, Hq, nblk]
    ok = ~osel.near                                                        # [B, R, Hq]
    assert np.array_equal(gk[ok], osel.kept[ok])
    assert ok.mean() > 0.95
    return gk


def check_tile_lists(sel, osel, C):
    """Needs osel over all rows 0..C-1."""
    B, _, Hq, nblk = osel.kept.shape
    tl = sel.tile_list.cpu().numpy()
    tc = sel.tile_cnt.cpu().numpy()
    n_qt = (C + 127) // 128
    for b in range(B):
        for h in range(Hq):
            for t in range(n_qt):
                rr = slice(t * 128, min(C, t * 128 + 128))
                if osel.near[b, rr, h].any():
                    continue
                expect = oracle.tile_union(osel.kept[b, rr, h])
                assert tc[b, h, t] == len(expect)
                assert np.array_equal(tl[b, h, t, :tc[b, h, t]], expect)


def run_sparse(w, s, C, alpha, rows=None):
    q = dev(w.q[:, s:s + C], w.dtype)
    k = dev(w.k[:, :s + C], w.dtype)
    v = dev(w.v[:, :s + C], w.dtype)
    sel = pfx.block_index(q, k, s, 128, alpha)
    pooled = pfx.alloc_pooled(q, k, s)
    out = pfx.attn_sparse(q, k, v, s, sel, pooled=pooled)
    pfx.stream_status()
    return q, k, v, sel, pooled, out


def ref_sparse(w, s, C, alpha, rows=None):
    q = w.f64(w.q[:, s:s + C])
    k = w.f64(w.k[:, :s + C])
    v = w.f64(w.v[:, :s + C])
    return oracle.sparse(q, k, v, s, 128, alpha, rows=rows)


@pytest.fixture(scope="module")
def small():
    return pi.planted_workload("sparse-small", 21, 1, 8, 2, 128, 2048, 2048, "bf16", beta=14.0)


@pytest.mark.parametrize("s,C", [(0, 2048), (1024, 1024), (768, 1000)])
def test_small_planted_selection_and_output(small, s, C):
    w = small
    C = min(C, w.N - s)
    q, k, v, sel, pooled, out = run_sparse(w, s, C, 0.1)
    ref, osel = ref_sparse(w, s, C, 0.1)
    check_selection(sel, osel, np.arange(C))
    check_tile_lists(sel, osel, C)
    # pooled keys and values are the fp32 block means
    kb = sel.kbar_mean.cpu().double().numpy()
    assert np.max(np.abs(kb - osel.kbar)) <= 1e-5
    vb = pfx.vbar_view(pooled, q, k, s).cpu().double().numpy()
    assert np.max(np.abs(vb - oracle.pool_blocks(w.f64(w.v[:, :s + C]), 128))) <= 1e-5
    ok = ~osel.near
    mx, mean = errors(out, ref)
    e = np.abs(out.cpu().double().numpy() - ref)[ok]
    assert e.max() <= MAX_ABS and e.mean() <= 5e-4, (e.max(), e.mean())
    assert oracle.skip_share(osel) > 0.5


def test_alpha_zero_equals_dense(small):
    w = small
    q, k, v, sel, _, out = run_sparse(w, 0, 2048, 0.0)
    dense = pfx.attn_dense(q, k[:, :0], v[:, :0], k, v, 0)
    pfx.stream_status()
    mx, _ = errors(out, dense.double().cpu().numpy())
    assert mx <= 2e-3
    ref = oracle.dense(w.f64(w.q), w.f64(w.k[:, :0]), w.f64(w.v[:, :0]), w.f64(w.k), w.f64(w.v), 0)
    assert_close(out, ref, "alpha 0")
    assert (sel.tile_cnt.cpu().numpy() == np.arange(1, 17)[None, None, :]).all()


def test_block_constant_keys_sparse_equals_dense():
    w = pi.planted_workload("const", 22, 1, 4, 2, 128, 1024, 1024, "bf16", beta=14.0)
    k = w.k.reshape(1, 8, 128, 2, 128)
    w.k = np.ascontiguousarray(np.broadcast_to(k[:, :, :1], k.shape).reshape(1, 1024, 2, 128))
    q, kd, vd, sel, _, out = run_sparse(w, 0, 1024, 0.1)
    ref = oracle.dense(w.f64(w.q), w.f64(w.k[:, :0]), w.f64(w.v[:, :0]), w.f64(w.k), w.f64(w.v), 0)
    assert_close(out, ref, "block-constant keys")


def test_negative_control(small):
    _, _, _, _, _, a = run_sparse(small, 0, 2048, 0.1)
    _, _, _, _, _, b = run_sparse(small, 0, 2048, 0.0)
    mx, _ = errors(a, b.double().cpu().numpy())
    assert mx >= 10 * MAX_ABS


@pytest.mark.slow
def test_config4_32k_sampled_rows():
    w = pi.config(4)
    C = w.N
    q, k, v, sel, _, out = run_sparse(w, 0, C, w.alpha)
    rows = sample_rows(C, 2048, 4)
    ref, osel = ref_sparse(w, 0, C, w.alpha, rows=rows)
    check_selection(sel, osel, rows)
    ok = ~osel.near
    e = np.abs(out[:, rows].cpu().double().numpy() - ref)[ok]
    assert e.max() <= MAX_ABS and e.mean() <= 5e-4, (e.max(), e.mean())
    # executed (tile-union) skip share of the planted workload
    tc = sel.tile_cnt.cpu().numpy().astype(np.float64)           # [1, Hq, nqt]
    cand = np.arange(tc.shape[-1])[None, None, :]
    share = 1 - ((tc - 1).sum() / max(1.0, cand.sum() * tc.shape[1]))
    assert 0.8 <= share <= 0.97, share


@pytest.mark.slow
def test_config5_128k_last_chunk_sampled_rows():
    w = pi.config(5)
    s = w.N - w.chunk
    C = w.chunk
    q, k, v, sel, _, out = run_sparse(w, s, C, w.alpha)
    rows = sample_rows(C, 512, 5)
    ref, osel = ref_sparse(w, s, C, w.alpha, rows=rows)
    check_selection(sel, osel, rows)
    ok = ~osel.near
    e = np.abs(out[:, rows].cpu().double().numpy() - ref)[ok]
    assert e.max() <= MAX_ABS and e.mean() <= 5e-4, (e.max(), e.mean())
    # and the dense 128K chunk on the same rows
    dq = q
    dense = pfx.attn_dense(dq, k[:, :s], v[:, :s], k[:, s:], v[:, s:], s)
    pfx.stream_status()
    dref = oracle.dense(w.f64(w.q[:, s:]), w.f64(w.k[:, :s]), w.f64(w.v[:, :s]), w.f64(w.k[:, s:]),
                        w.f64(w.v[:, s:]), s, rows=rows[:128])
    assert_close(dense[:, rows[:128]], dref, "dense 128K last chunk")


def test_sparse_lse_matches_oracle(small):
    """lse = log of the row's denominator (exact and pooled terms).  Exact keys: within
    1e-4 (fp32 scores and sums).  Pooled terms score q against kbar rounded to the input
    type (bf16: 2^-9 relative), and lse moves by at most the largest logit error, so with
    skipped blocks the bound adds 2^-9 * max |pooled logit|."""
    w = small
    s, C = 1024, 1024
    q = dev(w.q[:, s:s + C], w.dtype)
    k = dev(w.k[:, :s + C], w.dtype)
    v = dev(w.v[:, :s + C], w.dtype)
    for alpha in (0.0, 0.1):
        sel = pfx.block_index(q, k, s, 128, alpha)
        lse = torch.empty((1, q.shape[2], C), dtype=torch.float32, device="cuda")
        pfx.attn_sparse(q, k, v, s, sel, lse=lse)
        pfx.stream_status()
        _, osel, rlse = oracle.sparse(w.f64(w.q[:, s:s + C]), w.f64(w.k[:, :s + C]), w.f64(w.v[:, :s + C]),
                                      s, 128, alpha, with_lse=True)
        ok = ~osel.near
        got = lse.cpu().double().numpy().transpose(0, 2, 1)
        pooled_max = np.abs(np.where(np.isfinite(osel.scores), osel.scores, 0.0)).max()
        tol = 1e-4 if alpha == 0.0 else 1e-4 + 2.0 ** -9 * pooled_max
        assert np.max(np.abs(got - rlse)[ok]) <= tol, (alpha, np.max(np.abs(got - rlse)[ok]), tol)


# --------------------------------------------------------------------------- keep rules
RULES = [
    ("sinks-window", dict(sink_tokens=256, local_blocks=1)),
    ("tail", dict(dense_tail_rows=64)),
    ("row32", dict(row_group=32)),
    ("shared", dict(share_kv_group=1)),
    ("all", dict(sink_tokens=256, local_blocks=2, dense_tail_rows=64, row_group=32, share_kv_group=1)),
]


@pytest.mark.parametrize("name,kw", RULES)
def test_keep_rules_selection_and_output(small, name, kw):
    """Selection under the Metal port's keep rules: row bits and tile lists bit-exact with
    the oracle outside the near band (propagated through the group unions), outputs within
    tolerance."""
    w = small
    s, C = 1024, 1024
    q = dev(w.q[:, s:s + C], w.dtype)
    k = dev(w.k[:, :s + C], w.dtype)
    v = dev(w.v[:, :s + C], w.dtype)
    sel = pfx.block_index(q, k, s, 128, 0.1, rules=pf.KeepRules(**kw))
    out = pfx.attn_sparse(q, k, v, s, sel)
    pfx.stream_status()
    okw = dict(kw)
    okw["share_kv_group"] = bool(okw.get("share_kv_group", 0))
    ref, osel = oracle.sparse(w.f64(w.q[:, s:s + C]), w.f64(w.k[:, :s + C]), w.f64(w.v[:, :s + C]), s, 128,
                              0.1, rules=oracle.KeepRules(**okw))
    check_selection(sel, osel, np.arange(C))
    check_tile_lists(sel, osel, C)
    ok = ~osel.near
    e = np.abs(out.cpu().double().numpy() - ref)[ok]
    assert e.max() <= MAX_ABS and e.mean() <= 5e-4, (e.max(), e.mean())
