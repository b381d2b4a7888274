"""Block-sparse prefill through the C ABI against the float64 oracle: row selections equal
outside the 1e-4 threshold band (and inside it, differing only where rounding may decide a
pair either way), tile lists equal to the union of their rows, and every row's output within
tolerance, near-threshold rows included (their expected output follows the selection the GPU
took, which the oracle first checks is one the definition allows)."""
import numpy as np
import pytest
import torch

import oracle
import prefill_inputs as pi
from gpu_util import MAX_ABS, MEAN_ABS, assert_close, dev, errors, sample_rows
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


def expected_sparse(w, s, C, alpha, rows, sel, rules=None, with_lse=False):
    """The oracle's output on `rows` under the GPU's row selection, after checking that the
    selection equals the definition's outside the threshold band (ValueError otherwise).
    Returns (ref, osel, gk[, lse]) with gk the GPU's kept blocks [B, R, Hq, nblk]."""
    q = w.f64(w.q[:, s:s + C])
    k = w.f64(w.k[:, :s + C])
    v = w.f64(w.v[:, :s + C])
    nblk = (s + C + 127) // 128
    gk = gpu_bits_to_kept(sel.row_bits, nblk)[:, rows]
    r = oracle.sparse_for_selection(q, k, v, s, 128, alpha, gk, rows=rows, rules=rules, with_lse=with_lse)
    return (r[0], r[1], gk, r[3]) if with_lse else (r[0], r[1], gk)


def check_selection(osel, gk):
    """Row bits equal the definition's on every row outside the band; the band is rare."""
    ok = ~osel.near
    assert np.array_equal(gk[ok], osel.kept[ok])
    assert ok.mean() > 0.95


def check_tile_lists(sel, osel, C):
    """Every tile list is the ascending union of its rows' GPU row bits; on tiles without a
    near row it also equals the definition's union.  osel must cover rows 0..C-1."""
    B, _, Hq, nblk = osel.kept.shape
    gk = gpu_bits_to_kept(sel.row_bits, nblk)
    tl = sel.tile_list.cpu().numpy()
    tc = sel.tile_cnt.cpu().numpy()
    n_qt = (C + 127) // 128
    for b in range(B):
        for h in range(Hq):
            for t in range(n_qt):
                rr = slice(t * 128, min(C, t * 128 + 128))
                got = tl[b, h, t, :tc[b, h, t]]
                assert np.array_equal(got, oracle.tile_union(gk[b, rr, h]))
                if not osel.near[b, rr, h].any():
                    assert np.array_equal(got, oracle.tile_union(osel.kept[b, rr, h]))


def assert_rows_close(out, ref, what=""):
    e = np.abs(out.cpu().double().numpy() - ref)
    assert np.isfinite(e).all(), what
    print("%s: max abs error %.3g (%.0f%% of the bar), mean abs %.3g (%.0f%%)"
          % (what, e.max(), 100 * e.max() / MAX_ABS, e.mean(), 100 * e.mean() / MEAN_ABS))
    assert e.max() <= MAX_ABS and e.mean() <= MEAN_ABS, (what, e.max(), e.mean())


def run_sparse(w, s, C, alpha, rows=None):
    q = dev(w.q[:, s:s + C], w.dtype)
    k = dev(w.k[:, :s + C], w.dtype)
    v = dev(w.v[:, :s + C], w.dtype)
    sel = pfx.block_index(q, k, s, 128, alpha)
    pooled = pfx.alloc_pooled(q, k, s)
    out = pfx.attn_sparse(q, k, v, s, sel, pooled=pooled)
    pfx.stream_status()
    return q, k, v, sel, pooled, out


@pytest.fixture(scope="module")
def small():
    return pi.planted_workload("sparse-small", 21, 1, 8, 2, 128, 2048, 2048, "bf16", beta=14.0)


@pytest.mark.parametrize("s,C", [(0, 2048), (1024, 1024), (768, 1000)])
def test_small_planted_selection_and_output(small, s, C):
    w = small
    C = min(C, w.N - s)
    q, k, v, sel, pooled, out = run_sparse(w, s, C, 0.1)
    ref, osel, gk = expected_sparse(w, s, C, 0.1, np.arange(C), sel)
    check_selection(osel, gk)
    check_tile_lists(sel, osel, C)
    # pooled keys and values are the fp32 block means
    kb = sel.kbar_mean.cpu().double().numpy()
    assert np.max(np.abs(kb - osel.kbar)) <= 1e-5
    vb = pfx.vbar_view(pooled, q, k, s).cpu().double().numpy()
    assert np.max(np.abs(vb - oracle.pool_blocks(w.f64(w.v[:, :s + C]), 128))) <= 1e-5
    assert_rows_close(out, ref, "small planted")
    assert oracle.skip_share(osel) > 0.5


# shapes the block-sparse path takes besides the benchmark's: head dim 64, fp16 inputs, batch 2,
# and odd or unit query-head groups (one head per CTA at head dim 128, no head pairing)
SHAPES = [
    (2, 4, 2, 64, "f16", 512, 700),
    (1, 3, 1, 128, "bf16", 256, 900),
    (1, 2, 2, 128, "f16", 0, 1100),
    (2, 8, 2, 128, "bf16", 1024, 1024),
]


@pytest.mark.parametrize("B,Hq,Hkv,d,dtype,s,C", SHAPES)
def test_sparse_shapes_dtypes_and_batches(B, Hq, Hkv, d, dtype, s, C):
    """Selection (row bits and tile lists) and output against the oracle, every row of every
    batch and head, for a planted prompt of each shape; ragged chunks over a history."""
    w = pi.planted_workload("sparse-shape-%d-%d-%d-%d-%s" % (B, Hq, Hkv, d, dtype), 31 + d + Hq,
                            B, Hq, Hkv, d, s + C, C, dtype, beta=14.0)
    q, k, v, sel, pooled, out = run_sparse(w, s, C, 0.1)
    ref, osel, gk = expected_sparse(w, s, C, 0.1, np.arange(C), sel)
    check_selection(osel, gk)
    check_tile_lists(sel, osel, C)
    assert_rows_close(out, ref, "B %d Hq %d Hkv %d d %d %s" % (B, Hq, Hkv, d, dtype))
    assert oracle.skip_share(osel) > 0.3


def test_pipelined_chunks_equal_serial():
    """A chunked prompt with each chunk's block index on a low-priority stream ahead of the
    sparse attention on a high-priority stream (attention i waits for index i only; the pooled
    keys are shared and grow chunk by chunk): every chunk's output equals the one-stream run bit
    for bit, and the last chunk matches the oracle."""
    w = pi.planted_workload("pipelined", 33, 1, 8, 2, 128, 8192, 2048, "bf16", beta=14.0)
    N, C = w.N, w.chunk
    Q, K, V = dev(w.q, "bf16"), dev(w.k, "bf16"), dev(w.v, "bf16")
    starts = list(range(0, N, C))
    kbar = pfx.alloc_kbar(Q[:, :C], K, N, 128)
    pooled = pfx.alloc_pooled(Q[:, :C], K, 0, 128, max_keys=N)
    sels = [pfx.alloc_selection(Q[:, s:s + C], K[:, :s + C], s, 128, kbar=kbar, pooled_blocks=s // 128)
            for s in starts]
    outs = {m: torch.empty((len(starts), 1, C, 8, 128), dtype=torch.float32, device="cuda")
            for m in ("serial", "pipelined")}
    for i, s in enumerate(starts):
        pfx.block_index(Q[:, s:s + C], K[:, :s + C], s, 128, 0.1, sel=sels[i])
        pfx.attn_sparse(Q[:, s:s + C], K[:, :s + C], V[:, :s + C], s, sels[i], pooled=pooled,
                        out=outs["serial"][i])
    torch.cuda.synchronize()
    hi = torch.cuda.Stream(priority=-1)
    lo = torch.cuda.Stream(priority=0)
    start = torch.cuda.Event()
    start.record(torch.cuda.current_stream())
    hi.wait_event(start)
    lo.wait_event(start)
    for i, s in enumerate(starts):
        pfx.block_index(Q[:, s:s + C], K[:, :s + C], s, 128, 0.1, sel=sels[i], stream=lo)
        done = torch.cuda.Event()
        done.record(lo)
        hi.wait_event(done)
        pfx.attn_sparse(Q[:, s:s + C], K[:, :s + C], V[:, :s + C], s, sels[i], pooled=pooled,
                        out=outs["pipelined"][i], stream=hi)
    torch.cuda.synchronize()
    pfx.stream_status(hi)
    pfx.stream_status(lo)
    assert torch.equal(outs["serial"], outs["pipelined"])
    s = starts[-1]
    rows = sample_rows(C, 96, 34)
    ref, osel, gk = expected_sparse(w, s, C, 0.1, rows, sels[-1])
    check_selection(osel, gk)
    assert_rows_close(outs["pipelined"][-1][:, rows], ref, "pipelined last chunk")


def test_near_threshold_pairs_on_the_gpu(small):
    """alpha is set to one candidate's own probability ratio (rounded to fp32), so that pair --
    and any other within 1e-4 relative -- sits in the threshold band.  The GPU may decide it
    either way; its selection must differ from the definition's only there, and every row,
    the near ones included, must match the oracle under the selection the GPU took."""
    w = small
    s, C = 1024, 1024
    q64 = w.f64(w.q[:, s:s + C])
    k64 = w.f64(w.k[:, :s + C])
    rows = np.arange(C)
    probe = oracle.block_select(q64, k64, s, 128, 0.1, rows=rows[-128:], heads=[1])
    sc = probe.scores[0, 77, 0, :(s + rows[-128 + 77]) // 128]
    ratio = np.exp(sc - sc.max())
    alpha = float(np.float32(np.sort(ratio)[-2]))          # the second-hottest candidate
    q, k, v, sel, _, out = run_sparse(w, s, C, alpha)
    ref, osel, gk = expected_sparse(w, s, C, alpha, rows, sel)
    assert osel.near.sum() >= 1
    assert osel.near[0, C - 128 + 77, 1]
    check_tile_lists(sel, osel, C)
    assert_rows_close(out, ref, "near-threshold alpha %.9g" % alpha)
    near = osel.near
    e_near = np.abs(out.cpu().double().numpy() - ref)[near]
    assert e_near.max() <= MAX_ABS


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
def run_sparse_f16v(w, s, C, alpha):
    """As run_sparse, with v converted to fp16 first (the benchmark's configuration)."""
    q = dev(w.q[:, s:s + C], w.dtype)
    k = dev(w.k[:, :s + C], w.dtype)
    v = pfx.to_f16(dev(w.v[:, :s + C], w.dtype).contiguous())
    sel = pfx.block_index(q, k, s, 128, alpha)
    pooled = pfx.alloc_pooled(q, k, s)
    out = pfx.attn_sparse(q, k, v, s, sel, pooled=pooled)
    pfx.stream_status()
    return q, k, v, sel, pooled, out


def test_config4_32k_sampled_rows():
    """The 32K planted prompt in one call, as benchmarked (v kept in fp16)."""
    w = pi.config(4)
    C = w.N
    q, k, v, sel, _, out = run_sparse_f16v(w, 0, C, w.alpha)
    rows = sample_rows(C, 2048, 4)
    ref, osel, gk = expected_sparse(w, 0, C, w.alpha, rows, sel)
    check_selection(osel, gk)
    assert_rows_close(out[:, rows], ref, "32K sampled rows")
    # executed (tile-union) skip share of the planted workload
    tc = sel.tile_cnt.cpu().numpy().astype(np.float64)           # [1, Hq, nqt]
    cand = np.arange(tc.shape[-1])[None, None, :]
    share = 1 - ((tc - 1).sum() / max(1.0, cand.sum() * tc.shape[1]))
    assert 0.8 <= share <= 0.97, share


def test_sparse_lse_matches_oracle(small):
    """lse = log of the row's denominator (exact and pooled terms), on every row under the
    selection the GPU took.  Exact keys: within 1e-4 (fp32 scores and sums).  Pooled terms score q against kbar rounded to the input
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
        _, osel, _, rlse = expected_sparse(w, s, C, alpha, np.arange(C), sel, with_lse=True)
        got = lse.cpu().double().numpy().transpose(0, 2, 1)
        pooled_max = np.abs(np.where(np.isfinite(osel.scores), osel.scores, 0.0)).max()
        tol = 1e-4 if alpha == 0.0 else 1e-4 + 2.0 ** -9 * pooled_max
        assert np.max(np.abs(got - rlse)) <= tol, (alpha, np.max(np.abs(got - rlse)), tol)


def test_chunked_prompt_shares_pooled_blocks(small):
    """A prompt processed in chunks with one pooled-key buffer and one workspace for all of them
    (each call pools only the blocks the earlier chunks have not) gives bit-identical selections,
    pooled means and outputs to fresh buffers per chunk, and matches the oracle."""
    w = small
    N, CH = w.N, 512
    Q, K, V = dev(w.q, w.dtype), dev(w.k, w.dtype), dev(w.v, w.dtype)
    kbar = pfx.alloc_kbar(Q[:, :CH], K, N)
    pooled = pfx.alloc_pooled(Q[:, :CH], K, 0, max_keys=N)
    for s in range(0, N, CH):
        q, k, v = Q[:, s:s + CH], K[:, :s + CH], V[:, :s + CH]
        sel_r = pfx.alloc_selection(q, k, s, kbar=kbar, pooled_blocks=s // 128)
        pfx.block_index(q, k, s, 128, 0.1, sel=sel_r)
        out_r = pfx.attn_sparse(q, k, v, s, sel_r, pooled=pooled)
        sel_f = pfx.block_index(q, k, s, 128, 0.1)
        out_f = pfx.attn_sparse(q, k, v, s, sel_f)
        pfx.stream_status()
        nb = (s + CH + 127) // 128
        assert torch.equal(kbar[0][:, :, :nb], sel_f.kbar[0])
        assert torch.equal(sel_r.row_bits, sel_f.row_bits) and torch.equal(sel_r.tile_cnt, sel_f.tile_cnt)
        assert torch.equal(out_r, out_f)
    rows = np.arange(CH)
    ref, osel, gk = expected_sparse(w, N - CH, CH, 0.1, rows, sel_r)
    assert_rows_close(out_r, ref, "chunked with shared pooled blocks")


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
    the oracle outside the near band (propagated through the group unions), every row's
    output within tolerance."""
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
    ref, osel, gk = expected_sparse(w, s, C, 0.1, np.arange(C), sel, rules=oracle.KeepRules(**okw))
    check_selection(osel, gk)
    check_tile_lists(sel, osel, C)
    assert_rows_close(out, ref, "keep rules " + name)
