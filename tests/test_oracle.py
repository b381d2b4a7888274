"""Pins for the float64 oracle, each against something other than the oracle itself.

* brute force: per-element Python loops with math.exp on tiny inputs;
* closed forms and invariants: V = 1 gives 1; masked keys contribute exactly
  nothing; shift invariance of a fully masked row; chunked prefill equals
  one-shot causal prefill; GQA equals MHA over repeated K/V heads;
* the block-sparse path: alpha = 0 and block-constant keys reduce it to dense
  causal attention; a hand-worked 36-token toy fixes the selection and a
  hand-derived row fixes the pooled-correction weight n_b * e^(s_b) and vbar_b;
* the folded-indexer mask's visible-key budget 512*4 + 3 = 2051;
* the log-sum-exp output: identical keys give q.k0 * scale + log(visible count),
  a mask shift moves it by the same constant, results over disjoint key sets
  merge through it into the full result, and the toy's hand-derived
  denominator fixes the sparse one;
* the keep rules: the toy's golden lists extended by hand for sinks, a local
  window and a dense tail, hand-worked unions for 2-row groups and for a KV
  group of two query heads, sharing as a no-op without groups, and dense-tail
  rows reducing to plain causal attention.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import prefill_inputs as pi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_dense_row(qi, keys, vals, mrow, scale):
    """softmax((q.k) * scale + M) V for one query row, plain loops."""
    logits = []
    for j in range(len(keys)):
        dot = 0.0
        for a in range(len(qi)):
            dot += qi[a] * keys[j][a]
        logits.append(dot * scale + mrow[j])
    mx = max(logits)
    w = [math.exp(x - mx) for x in logits]
    z = math.fsum(w)
    return [math.fsum(w[j] * vals[j][a] for j in range(len(keys))) / z for a in range(len(vals[0]))]


def rand_case(seed, B=2, Hq=4, Hkv=2, C=5, s=3, d=8):
    g = np.random.default_rng(seed)
    q = g.standard_normal((B, C, Hq, d))
    kh, vh = g.standard_normal((B, s, Hkv, d)), g.standard_normal((B, s, Hkv, d))
    kc, vc = g.standard_normal((B, C, Hkv, d)), g.standard_normal((B, C, Hkv, d))
    return q, kh, vh, kc, vc


@pytest.mark.parametrize("masked", [False, True])
def test_dense_matches_brute_force(masked):
    q, kh, vh, kc, vc = rand_case(1)
    B, C, Hq, d = q.shape
    s, Hkv = kh.shape[1], kh.shape[2]
    T = s + C
    g = np.random.default_rng(2)
    if masked:
        mask = g.uniform(-3.0, 0.0, size=(C, T))
        mask[g.random((C, T)) < 0.3] = -30000.0
        mask[:, 0] = -1.0  # every row keeps a visible key
    else:
        mask = None
    scale = 0.37
    out = oracle.dense(q, kh, vh, kc, vc, s, mask=mask, scale=scale)
    k = np.concatenate([kh, kc], 1)
    v = np.concatenate([vh, vc], 1)
    for b in range(B):
        for h in range(Hq):
            gg = h // (Hq // Hkv)
            for i in range(C):
                if mask is None:
                    mrow = [0.0 if j <= s + i else -30000.0 for j in range(T)]
                else:
                    mrow = list(mask[i])
                ref = brute_dense_row(list(q[b, i, h]), k[b, :, gg].tolist(), v[b, :, gg].tolist(), mrow, scale)
                assert np.max(np.abs(out[b, i, h] - ref)) <= 1e-12


def test_default_scale_is_inverse_sqrt_d():
    q, kh, vh, kc, vc = rand_case(3)
    d = q.shape[-1]
    a = oracle.dense(q, kh, vh, kc, vc, kh.shape[1])
    b = oracle.dense(q, kh, vh, kc, vc, kh.shape[1], scale=1.0 / math.sqrt(d))
    assert np.array_equal(a, b)


def test_ones_value_gives_one():
    q, kh, vh, kc, vc = rand_case(4)
    out = oracle.dense(q, kh, np.ones_like(vh), kc, np.ones_like(vc), kh.shape[1])
    assert np.max(np.abs(out - 1.0)) <= 1e-12


def test_masked_key_contributes_exactly_zero():
    q, kh, vh, kc, vc = rand_case(5, C=6, s=4)
    C, s = q.shape[1], kh.shape[1]
    g = np.random.default_rng(6)
    mask = np.where(g.random((C, s + C)) < 0.5, -30000.0, 0.0)
    mask[:, 1] = 0.0
    base = oracle.dense(q, kh, vh, kc, vc, s, mask=mask)
    # perturb V of a key that every row masks; the output must not move a single bit
    mask[:, 2] = -30000.0
    base = oracle.dense(q, kh, vh, kc, vc, s, mask=mask)
    vh2 = vh.copy()
    vh2[:, 2] += 1e3
    pert = oracle.dense(q, kh, vh2, kc, vc, s, mask=mask)
    assert np.array_equal(base, pert)


def test_fully_masked_row_is_plain_softmax():
    """A row whose every key carries -30000 is shift-invariant: it equals the unmasked row."""
    q, kh, vh, kc, vc = rand_case(7, C=4, s=4)
    C, s = q.shape[1], kh.shape[1]
    mask = np.zeros((C, s + C))
    mask[2, :] = -30000.0
    a = oracle.dense(q, kh, vh, kc, vc, s, mask=mask)
    b = oracle.dense(q, kh, vh, kc, vc, s, mask=np.zeros((C, s + C)))
    assert np.max(np.abs(a[:, 2] - b[:, 2])) <= 1e-9
    assert np.array_equal(a[:, [0, 1, 3]], b[:, [0, 1, 3]])


def test_explicit_causal_mask_equals_default():
    q, kh, vh, kc, vc = rand_case(8, C=7, s=5)
    C, s = q.shape[1], kh.shape[1]
    a = oracle.dense(q, kh, vh, kc, vc, s)
    b = oracle.dense(q, kh, vh, kc, vc, s, mask=pi.causal_mask(C, s, np.float64))
    assert np.array_equal(a, b)


def test_chunked_equals_one_shot():
    """Chunks at start 0, 64, 128 over the previous chunks' K/V equal one causal pass over 192 rows."""
    g = np.random.default_rng(9)
    B, Hq, Hkv, d, N, C = 1, 4, 2, 16, 192, 64
    q = g.standard_normal((B, N, Hq, d))
    k = g.standard_normal((B, N, Hkv, d))
    v = g.standard_normal((B, N, Hkv, d))
    one = oracle.dense(q, k[:, :0], v[:, :0], k, v, 0)
    for s in range(0, N, C):
        part = oracle.dense(q[:, s:s + C], k[:, :s], v[:, :s], k[:, s:s + C], v[:, s:s + C], s)
        assert np.max(np.abs(part - one[:, s:s + C])) <= 1e-12


def test_gqa_equals_repeated_kv_heads():
    q, kh, vh, kc, vc = rand_case(10, Hq=6, Hkv=2)
    s = kh.shape[1]
    a = oracle.dense(q, kh, vh, kc, vc, s)
    rep = lambda x: np.repeat(x, 3, axis=2)  # head h of 6 reads KV head h // 3
    b = oracle.dense(q, rep(kh), rep(vh), rep(kc), rep(vc), s)
    assert np.max(np.abs(a - b)) <= 1e-15


def test_rows_and_heads_subsets_agree():
    q, kh, vh, kc, vc = rand_case(11, C=9, s=6)
    s = kh.shape[1]
    full = oracle.dense(q, kh, vh, kc, vc, s)
    sub = oracle.dense(q, kh, vh, kc, vc, s, rows=[8, 1, 4], heads=[3, 0])
    assert np.array_equal(sub, full[:, [8, 1, 4]][:, :, [3, 0]])


def test_cache_layout_is_a_relayout():
    _, _, _, kc, _ = rand_case(12)
    lay = oracle.chunk_kv_cache_layout(kc)
    B, C, H, d = kc.shape
    for b in range(B):
        for h in range(H):
            for t in range(C):
                assert np.array_equal(lay[b, h, t], kc[b, t, h])


# --------------------------------------------------------------------------
# folded indexer mask (the generator's budget)
# --------------------------------------------------------------------------
def test_folded_mask_visible_budget():
    """ANE Prefill Research, 'Folding a sparse indexer's selection': keptBlocks*ratio + (ratio-1) = 2051."""
    s, C = 2048, 64
    mask, kept = pi.indexer_fold_mask(77, C, s)
    counts = (mask == 0.0).sum(axis=1)
    p = s + np.arange(C)
    assert np.array_equal(counts, 512 * 4 + (p + 1) % 4)
    assert counts.max() == 512 * 4 + (4 - 1) == 2051
    for i in range(C):
        assert kept[i][-1] == (s + i + 1) // 4 - 1          # newest complete block always kept
        assert len(set(kept[i].tolist())) == 512
        assert np.all(mask[i, s + i + 1:] == -30000.0)      # no future key is visible


# --------------------------------------------------------------------------
# index-driven attention (the indexer's keep lists, gathered)
# --------------------------------------------------------------------------
def _visible_by_predicate(p, kept, ratio):
    """Key j is visible iff its compressed block is kept and complete, or j lies after the
    last complete block and not after p (a membership test, not the oracle's construction)."""
    n_complete = (p + 1) // ratio
    kept = set(int(c) for c in kept)
    return [j for j in range(p + 1)
            if (j // ratio in kept and j // ratio < n_complete) or n_complete * ratio <= j <= p]


@pytest.mark.parametrize("ratio", [3, 4])
def test_indexed_matches_brute_force_over_the_visible_keys(ratio):
    q, kh, vh, kc, vc = rand_case(11, B=1, Hq=4, Hkv=2, C=6, s=12, d=8)
    B, C, Hq, d = q.shape
    s = kh.shape[1]
    g = np.random.default_rng(12)
    kept = [g.choice((s + i + 1) // ratio, size=min(2, (s + i + 1) // ratio), replace=False)
            for i in range(C)]
    out = oracle.dense_indexed(q, kh, vh, kc, vc, s, kept, ratio)
    k = np.concatenate([kh, kc], axis=1)
    v = np.concatenate([vh, vc], axis=1)
    for i in range(C):
        js = _visible_by_predicate(s + i, kept[i], ratio)
        for h in range(Hq):
            gk = h // (Hq // kh.shape[2])
            ref = brute_dense_row(q[0, i, h], [k[0, j, gk] for j in js], [v[0, j, gk] for j in js],
                                  [0.0] * len(js), 1.0 / math.sqrt(d))
            assert np.max(np.abs(out[0, i, h] - ref)) < 1e-12


def test_indexed_equals_the_folded_mask():
    """The pages fold the same selection into an additive mask at -30000: same result."""
    s, C, ratio, nk = 256, 64, 4, 16
    q, kh, vh, kc, vc = rand_case(13, B=1, Hq=4, Hkv=2, C=C, s=s, d=16)
    mask, kept = pi.indexer_fold_mask(14, C, s, kept_blocks=nk, ratio=ratio)
    a = oracle.dense(q, kh, vh, kc, vc, s, mask=mask.astype(np.float64))
    b = oracle.dense_indexed(q, kh, vh, kc, vc, s, kept, ratio)
    assert np.max(np.abs(a - b)) < 1e-12


def test_indexed_all_complete_blocks_is_causal():
    s, C, ratio = 20, 9, 4
    q, kh, vh, kc, vc = rand_case(15, B=2, Hq=2, Hkv=1, C=C, s=s, d=8)
    kept = [np.arange((s + i + 1) // ratio) for i in range(C)]
    a = oracle.dense(q, kh, vh, kc, vc, s)
    b = oracle.dense_indexed(q, kh, vh, kc, vc, s, kept, ratio)
    assert np.max(np.abs(a - b)) < 1e-12


@pytest.mark.parametrize("ratio", [3, 4, 5])
def test_indexed_visible_count(ratio):
    """keptBlocks x ratio + ((p + 1) mod ratio) keys; duplicates and order change nothing."""
    g = np.random.default_rng(16)
    for p in range(40, 60):
        nc = (p + 1) // ratio
        kept = g.choice(nc, size=5, replace=False)
        vis = oracle.indexed_visible_keys(p, kept, ratio)
        assert len(vis) == 5 * ratio + (p + 1) % ratio
        assert vis.max() <= p
        dup = np.concatenate([kept[::-1], kept[:2]])
        assert np.array_equal(oracle.indexed_visible_keys(p, dup, ratio), vis)


def test_indexed_negative_control():
    """The pages' check that was not sensitive enough: a causal-only run must differ from the
    selection by far more than the parity tolerance, or a test comparing them proves nothing."""
    s, C, ratio, nk = 512, 32, 4, 16
    q, kh, vh, kc, vc = rand_case(19, B=1, Hq=2, Hkv=1, C=C, s=s, d=32)
    _, kept = pi.indexer_fold_mask(20, C, s, kept_blocks=nk, ratio=ratio)
    sel = oracle.dense_indexed(q, kh, vh, kc, vc, s, kept, ratio)
    causal = oracle.dense(q, kh, vh, kc, vc, s)
    assert np.max(np.abs(sel - causal)) >= 10 * 5e-3


def test_indexed_rejects_a_bad_selection():
    with pytest.raises(ValueError):
        oracle.indexed_visible_keys(10, [2], 4)       # block 2 holds keys 8..11: not complete at 10
    with pytest.raises(ValueError):
        oracle.indexed_visible_keys(10, [-1], 4)
    with pytest.raises(ValueError):
        oracle.indexed_visible_keys(11, [], 4)        # 12 keys in 3 complete blocks, none kept
    assert list(oracle.indexed_visible_keys(10, [], 4)) == [8, 9, 10]


def test_indexed_single_key_returns_its_value_and_lse():
    """A row whose only visible key is its own (p + 1 = 1 mod ratio, nothing kept): out = v_p,
    lse = (q . k_p) * scale."""
    s, C, ratio = 8, 1, 4                              # p = 8: tail = key 8 alone
    q, kh, vh, kc, vc = rand_case(17, B=1, Hq=2, Hkv=2, C=C, s=s, d=8)
    out, lse = oracle.dense_indexed(q, kh, vh, kc, vc, s, [np.array([], dtype=np.int64)], ratio,
                                    with_lse=True)
    assert np.array_equal(out[0, 0], vc[0, 0])
    for h in range(2):
        assert abs(lse[0, 0, h] - float(q[0, 0, h] @ kc[0, 0, h]) / math.sqrt(8)) < 1e-12


def test_indexed_lse_identical_keys_closed_form():
    """All keys equal: lse = log(visible count) + (q . k) * scale."""
    s, C, ratio = 16, 4, 4
    q, kh, vh, kc, vc = rand_case(18, B=1, Hq=1, Hkv=1, C=C, s=s, d=4)
    kh[:] = 0.25
    kc[:] = 0.25
    kept = [np.array([0, 2]), np.array([1]), np.array([], dtype=np.int64), np.array([0, 1, 3])]
    _, lse = oracle.dense_indexed(q, kh, vh, kc, vc, s, kept, ratio, with_lse=True)
    for i in range(C):
        n = len(kept[i]) * ratio + (s + i + 1) % ratio
        assert abs(lse[0, i, 0] - (math.log(n) + q[0, i, 0].sum() * 0.25 / 2.0)) < 1e-12


# --------------------------------------------------------------------------
# block-sparse path
# --------------------------------------------------------------------------
def toy36(e_scale=1.0):
    cfg = json.load(open(os.path.join(GOLDEN, "toy36.json")))["construction"]
    N, blk, d = cfg["N"], cfg["block"], cfg["d"]
    t = cfg["t"]
    q = np.zeros((1, N, 1, d))
    q[0, :, 0, :] = cfg["q_row"]
    k = np.zeros((1, N, 1, d))
    v = np.zeros((1, N, 1, d))
    for j in range(N):
        e = (0.5 if j % 2 == 0 else -0.5) * e_scale
        k[0, j, 0, 0] = t[j // blk] + e
        v[0, j, 0] = (1.0, e, j // blk, 0.0)
    return q, k, v, blk, cfg["scale"]


@pytest.mark.parametrize("alpha", ["0.2", "0.1", "0.0"])
def test_toy36_selection(alpha):
    gold = json.load(open(os.path.join(GOLDEN, "toy36.json")))
    q, k, v, blk, scale = toy36()
    sel = oracle.block_select(q, k, 0, blk, float(alpha), scale=scale)
    assert np.allclose(sel.kbar[0, 0, :, 0], gold["construction"]["t"])
    for qb, expect in enumerate(gold["kept_by_query_block"][alpha]):
        for r in range(qb * blk, (qb + 1) * blk):
            assert np.flatnonzero(sel.kept[0, r, 0]).tolist() == expect
        assert oracle.tile_union(sel.kept[0, qb * blk:(qb + 1) * blk, 0]).tolist() == expect
    assert not sel.near.any()
    n_off = sum(len(e) - 1 for e in gold["kept_by_query_block"][alpha]) * blk
    assert n_off == gold["kept_offdiag_pairs"][alpha]
    assert abs(oracle.skip_share(sel) - (1 - n_off / gold["candidate_pairs"])) < 1e-12


def test_toy36_pooled_correction_closed_form():
    """Row 12 of the toy at alpha 0.2, derived by hand.

    Kept {1, 2}, skipped {0}.  Exact logits: block 1 keys 3 +- 0.5 (three each),
    key 12 (block 2) 1 + 0.5; block 0 is represented by one pooled logit t_0 = 0
    with weight n_0 = 6 and value vbar_0 = (1, 0, 0, 0).
    """
    q, k, v, blk, scale = toy36()
    out, _ = oracle.sparse(q, k, v, 0, blk, 0.2, scale=scale, rows=[12])
    e35, e25, e15 = math.exp(3.5), math.exp(2.5), math.exp(1.5)
    den = 3 * e35 + 3 * e25 + e15 + 6 * math.exp(0.0)
    expect = [1.0,
              (3 * e35 * 0.5 - 3 * e25 * 0.5 + e15 * 0.5 + 6 * 0.0) / den,
              ((3 * e35 + 3 * e25) * 1 + e15 * 2 + 6 * 0.0) / den,
              0.0]
    assert np.max(np.abs(out[0, 0, 0] - expect)) <= 1e-14
    # the dense row differs (block 0 exact: logits +-0.5) -- the correction is live
    dense = oracle.dense(q, k[:, :0], v[:, :0], k, v, 0, scale=scale, rows=[12])
    assert np.max(np.abs(dense[0, 0, 0] - out[0, 0, 0])) > 1e-3


def test_toy36_without_spread_sparse_equals_dense():
    q, k, v, blk, scale = toy36(e_scale=0.0)
    dense = oracle.dense(q, k[:, :0], v[:, :0], k, v, 0, scale=scale)
    for alpha in (0.2, 0.1, 1.0):
        out, _ = oracle.sparse(q, k, v, 0, blk, alpha, scale=scale)
        assert np.max(np.abs(out - dense)) <= 1e-12


def sparse_case(seed, N=80, s=16, Hq=4, Hkv=2, d=8):
    g = np.random.default_rng(seed)
    q = g.standard_normal((1, N, Hq, d))
    k = g.standard_normal((1, s + N, Hkv, d))
    v = g.standard_normal((1, s + N, Hkv, d))
    return q, k, v, s


def test_sparse_alpha_zero_equals_dense():
    q, k, v, s = sparse_case(20)
    dense = oracle.dense(q, k[:, :s], v[:, :s], k[:, s:], v[:, s:], s)
    out, sel = oracle.sparse(q, k, v, s, 8, 0.0)
    assert oracle.skip_share(sel) == 0.0
    assert np.max(np.abs(out - dense)) <= 1e-12


def test_sparse_block_constant_keys_equals_dense():
    """Keys constant within each block make the pooled row exact: sparse == dense for every alpha."""
    q, k, v, s = sparse_case(21)
    blk = 8
    T = k.shape[1]
    for b0 in range(0, T, blk):
        k[:, b0:b0 + blk] = k[:, b0:b0 + 1]
    dense = oracle.dense(q, k[:, :s], v[:, :s], k[:, s:], v[:, s:], s)
    for alpha in (0.05, 0.3, 0.9, 1.0):
        out, sel = oracle.sparse(q, k, v, s, blk, alpha)
        assert oracle.skip_share(sel) > 0.0
        assert np.max(np.abs(out - dense)) <= 1e-12


def test_sparse_single_block_equals_dense():
    q, k, v, _ = sparse_case(22, N=7, s=0)
    dense = oracle.dense(q, k[:, :0], v[:, :0], k, v, 0)
    out, _ = oracle.sparse(q, k, v, 0, 8, 0.5)
    assert np.max(np.abs(out - dense)) <= 1e-12


def test_pool_blocks_against_prefix_sums():
    g = np.random.default_rng(23)
    x = g.standard_normal((2, 29, 3, 5))
    pooled = oracle.pool_blocks(x, 8)
    cs = np.concatenate([np.zeros((2, 1, 3, 5)), np.cumsum(x, axis=1)], axis=1)
    for bk in range(4):
        a, e = bk * 8, min(29, bk * 8 + 8)
        assert np.allclose(pooled[:, :, bk], ((cs[:, e] - cs[:, a]) / (e - a)), atol=1e-13)
    assert np.array_equal(oracle.block_counts(29, 8), [8, 8, 8, 5])


def test_selection_nested_in_alpha():
    q, k, v, s = sparse_case(24, N=120, s=40)
    sels = [oracle.block_select(q, k, s, 8, a) for a in (1.0, 0.5, 0.1, 0.0)]
    for lo, hi in zip(sels, sels[1:]):
        assert np.all(~lo.kept | hi.kept)
    # alpha = 1 keeps the diagonal plus the hottest candidate(s) only
    sel = sels[0]
    ob = (s + sel.rows) // 8
    for r in range(len(sel.rows)):
        for hi_ in range(q.shape[2]):
            kept = set(np.flatnonzero(sel.kept[0, r, hi_]).tolist())
            if ob[r] == 0:
                assert kept == {0}
            else:
                best = int(np.argmax(sel.scores[0, r, hi_, :ob[r]]))
                assert kept == {best, int(ob[r])}


def test_sparse_negative_control():
    """alpha 0.1 vs alpha 0 on planted data must differ by >= 10x the 5e-3 output tolerance."""
    w = pi.planted_workload("tiny", 5, 1, 4, 2, 32, 1024, 1024, "bf16", block=64, beta=8.0)
    q, k, v = w.f64(w.q), w.f64(w.k), w.f64(w.v)
    rows = np.arange(512, 1024, 7)
    a, sel = oracle.sparse(q, k, v, 0, 64, 0.1, rows=rows)
    b, _ = oracle.sparse(q, k, v, 0, 64, 0.0, rows=rows)
    assert oracle.skip_share(sel) > 0.5
    assert np.max(np.abs(a - b)) > 10 * 5e-3


# --------------------------------------------------------------------------- log-sum-exp
def test_lse_identical_keys_closed_form():
    """Every key equal to k0: row i sees s + i + 1 keys, so lse = q.k0 * scale + log(s + i + 1)."""
    g = np.random.default_rng(40)
    B, C, s, Hq, Hkv, d = 1, 6, 5, 2, 1, 8
    q = g.standard_normal((B, C, Hq, d))
    k0 = g.standard_normal(d)
    kh = np.broadcast_to(k0, (B, s, Hkv, d)).copy()
    kc = np.broadcast_to(k0, (B, C, Hkv, d)).copy()
    v = g.standard_normal((B, s + C, Hkv, d))
    _, lse = oracle.dense(q, kh, v[:, :s], kc, v[:, s:], s, with_lse=True)
    scale = 1.0 / math.sqrt(d)
    for i in range(C):
        for h in range(Hq):
            assert abs(lse[0, i, h] - (float(q[0, i, h] @ k0) * scale + math.log(s + i + 1))) <= 1e-12


def test_lse_shifts_with_the_mask():
    q, kh, vh, kc, vc = rand_case(41)
    C, s = q.shape[1], kh.shape[1]
    mask = np.where(np.random.default_rng(42).random((C, s + C)) < 0.3, -30000.0, 0.0)
    out0, lse0 = oracle.dense(q, kh, vh, kc, vc, s, mask=mask, with_lse=True)
    out1, lse1 = oracle.dense(q, kh, vh, kc, vc, s, mask=mask + 2.5, with_lse=True)
    assert np.max(np.abs(lse1 - lse0 - 2.5)) <= 1e-12
    assert np.max(np.abs(out1 - out0)) <= 1e-12


def test_lse_merges_disjoint_key_sets():
    """Split-KV identity: attention over history and over the chunk separately, merged
    through their log-sum-exps, is attention over both."""
    q, kh, vh, kc, vc = rand_case(43)
    C, s = q.shape[1], kh.shape[1]
    full, lse = oracle.dense(q, kh, vh, kc, vc, s, with_lse=True)
    causal = oracle.causal_additive(C, s)
    hist_only = causal.copy()
    hist_only[:, s:] = -30000.0
    chunk_only = causal.copy()
    chunk_only[:, :s] = -30000.0
    oa, la = oracle.dense(q, kh, vh, kc, vc, s, mask=hist_only, with_lse=True)
    ob, lb = oracle.dense(q, kh, vh, kc, vc, s, mask=chunk_only, with_lse=True)
    merged_lse = np.logaddexp(la, lb)
    merged = (np.exp(la - merged_lse)[..., None] * oa + np.exp(lb - merged_lse)[..., None] * ob)
    assert np.max(np.abs(merged_lse - lse)) <= 1e-12
    assert np.max(np.abs(merged - full)) <= 1e-12


def test_sparse_lse_toy36_closed_form():
    """Row 12 of the toy (kept {1, 2}, block 0 pooled with weight 6 and logit 0): the
    denominator is 3e^3.5 + 3e^2.5 + e^1.5 + 6."""
    q, k, v, blk, scale = toy36()
    _, _, lse = oracle.sparse(q, k, v, 0, blk, 0.2, scale=scale, rows=[12], with_lse=True)
    den = 3 * math.exp(3.5) + 3 * math.exp(2.5) + math.exp(1.5) + 6.0
    assert abs(lse[0, 0, 0] - math.log(den)) <= 1e-13


def test_sparse_lse_alpha_zero_equals_dense():
    q, k, v, s = sparse_case(44)
    _, dlse = oracle.dense(q, k[:, :s], v[:, :s], k[:, s:], v[:, s:], s, with_lse=True)
    _, _, slse = oracle.sparse(q, k, v, s, 8, 0.0, with_lse=True)
    assert np.max(np.abs(slse - dlse)) <= 1e-12


# --------------------------------------------------------------------------- keep rules
def _toy_kept(sel, blk=6, head=0):
    return [np.flatnonzero(sel.kept[0, qb * blk, head]).tolist() for qb in range(6)]


def test_keep_rules_off_equal_the_base_rule():
    q, k, v, s = sparse_case(50)
    a = oracle.block_select(q, k, s, 8, 0.1)
    b = oracle.block_select(q, k, s, 8, 0.1, rules=oracle.KeepRules())
    assert np.array_equal(a.kept, b.kept)


def test_toy36_sinks_window_and_tail_by_hand():
    """From the alpha 0.2 golden lists: a 6-token sink adds block 0, a one-block window
    adds block qb-1, a 6-row dense tail makes the last query block keep every candidate."""
    q, k, v, blk, scale = toy36()
    sink = oracle.block_select(q, k, 0, blk, 0.2, scale=scale, rules=oracle.KeepRules(sink_tokens=6))
    assert _toy_kept(sink) == [[0], [0, 1], [0, 1, 2], [0, 1, 3], [0, 1, 3, 4], [0, 1, 3, 5]]
    win = oracle.block_select(q, k, 0, blk, 0.2, scale=scale, rules=oracle.KeepRules(local_blocks=1))
    assert _toy_kept(win) == [[0], [0, 1], [1, 2], [1, 2, 3], [1, 3, 4], [1, 3, 4, 5]]
    tail = oracle.block_select(q, k, 0, blk, 0.2, scale=scale, rules=oracle.KeepRules(dense_tail_rows=6))
    assert _toy_kept(tail) == [[0], [0, 1], [1, 2], [1, 3], [1, 3, 4], [0, 1, 2, 3, 4, 5]]
    assert np.flatnonzero(tail.kept[0, 29, 0]).tolist() == [1, 3, 4]   # row 29 is not in the tail


def _toy_two_signs():
    """The toy's keys with two queries: +(2,0,0,0) scores the blocks t_b, -(2,0,0,0) scores
    -t_b = (0, -3, -1, -2.5, -0.5, 1).  At alpha 0.2, in query block 4 (candidates 0..3) the
    first keeps {1, 3} (t >= 3 - 1.609) and the second keeps {0, 2} (-t >= 0 - 1.609)."""
    q, k, v, blk, scale = toy36()
    q2 = np.concatenate([q, -q], axis=2)                      # two query heads, one KV head
    return q2, k, v, blk, scale


def test_rows_grouped_take_the_union_by_hand():
    q2, k, v, blk, scale = _toy_two_signs()
    q = q2.copy()
    q[0, 25, 0] = -q2[0, 25, 0]                              # row 25 of head 0 scores -t_b
    sel = oracle.block_select(q[:, :, :1], k, 0, blk, 0.2, scale=scale)
    assert np.flatnonzero(sel.kept[0, 24, 0]).tolist() == [1, 3, 4]
    assert np.flatnonzero(sel.kept[0, 25, 0]).tolist() == [0, 2, 4]
    grp = oracle.block_select(q[:, :, :1], k, 0, blk, 0.2, scale=scale,
                              rules=oracle.KeepRules(row_group=2))
    for r in (24, 25):
        assert np.flatnonzero(grp.kept[0, r, 0]).tolist() == [0, 1, 2, 3, 4]
    assert np.flatnonzero(grp.kept[0, 26, 0]).tolist() == [1, 3, 4]      # rows 26, 27 untouched


def test_kv_group_shares_the_union_by_hand():
    q2, k, v, blk, scale = _toy_two_signs()
    alone = oracle.block_select(q2, k, 0, blk, 0.2, scale=scale)
    assert np.flatnonzero(alone.kept[0, 24, 1]).tolist() == [0, 2, 4]
    shared = oracle.block_select(q2, k, 0, blk, 0.2, scale=scale,
                                 rules=oracle.KeepRules(share_kv_group=True))
    for h in (0, 1):
        assert np.flatnonzero(shared.kept[0, 24, h]).tolist() == [0, 1, 2, 3, 4]


def test_kv_group_sharing_is_a_no_op_without_groups():
    q, k, v, s = sparse_case(51, Hq=2, Hkv=2)
    a = oracle.block_select(q, k, s, 8, 0.1)
    b = oracle.block_select(q, k, s, 8, 0.1, rules=oracle.KeepRules(share_kv_group=True))
    assert np.array_equal(a.kept, b.kept)


def test_dense_tail_rows_equal_dense_attention():
    """Rows in the dense tail keep every candidate, so their sparse output is plain causal
    attention (no pooled term)."""
    q, k, v, s = sparse_case(52)
    N = q.shape[1]
    out, _ = oracle.sparse(q, k, v, s, 8, 0.1, rules=oracle.KeepRules(dense_tail_rows=16))
    dense = oracle.dense(q, k[:, :s], v[:, :s], k[:, s:], v[:, s:], s)
    assert np.max(np.abs(out[0, N - 16:] - dense[0, N - 16:])) <= 1e-12
    assert np.max(np.abs(out[0, :N - 16] - dense[0, :N - 16])) > 1e-6    # the rest is sparse


# --------------------------------------------------------------------------
# the near-threshold band: pairs whose probability ratio sits within 1e-4 relative of alpha
# --------------------------------------------------------------------------
def _band_case(eps, alpha=0.1, t3=10.0, spread=0.0):
    """Four 2-token blocks of keys (t_b, 0, 0, 0), query (1, 0, 0, 0), scale 1, so the pooled
    logit of block b is exactly t_b.  Rows 6 and 7 (block 3) have candidates 0, 1, 2:
    t_0 = 0 is the hottest candidate, t_1 = ln(alpha (1 + eps)) puts block 1's probability
    ratio at alpha (1 + eps), t_2 = -5 is far below the threshold; the diagonal block 3 has
    t_3 (default 10, above every candidate: it must not enter the row maximum).  Rows 4 and 5
    (block 2) have candidates 0 and 1 against the same maximum.  With spread, the keys of
    every block alternate t_b + spread, t_b - spread (the block mean stays t_b)."""
    t = [0.0, math.log(alpha * (1.0 + eps)), -5.0, t3]
    N, blk, d = 8, 2, 4
    q = np.zeros((1, N, 1, d))
    q[0, :, 0, 0] = 1.0
    k = np.zeros((1, N, 1, d))
    v = np.zeros((1, N, 1, d))
    for j in range(N):
        k[0, j, 0, 0] = t[j // blk] + (spread if j % 2 == 0 else -spread)
        v[0, j, 0] = (1.0, j, (j % 2) - 0.5, j // blk)
    return q, k, v, blk, t


@pytest.mark.parametrize("eps", [5e-5, -5e-5, 9e-5, -9e-5])
def test_near_band_flags_a_pair_inside(eps):
    q, k, v, blk, _ = _band_case(eps)
    sel = oracle.block_select(q, k, 0, blk, 0.1, scale=1.0)
    for r in (4, 5, 6, 7):                           # blocks 2 and 3: block 1 is a candidate
        assert sel.near[0, r, 0]
        assert np.flatnonzero(sel.near_pairs[0, r, 0]).tolist() == [1]
    assert not sel.near[0, :4].any()
    # inside the band the definition still decides by >=: kept iff the ratio >= alpha
    assert bool(sel.kept[0, 6, 0, 1]) == (eps >= 0)


@pytest.mark.parametrize("eps", [5e-3, -5e-3, 5e-4, -5e-4, 1.5e-4, -1.5e-4])
def test_near_band_silent_outside(eps):
    """Outside 1e-4 relative the flag stays silent; +-5e-4 relative is only 5e-5 absolute at
    alpha 0.1, so an absolute band of 1e-4 would fire there."""
    q, k, v, blk, _ = _band_case(eps)
    sel = oracle.block_select(q, k, 0, blk, 0.1, scale=1.0)
    assert not sel.near.any()
    assert not sel.near_pairs.any()
    assert bool(sel.kept[0, 6, 0, 1]) == (eps > 0)


def test_near_band_scales_with_alpha():
    """The band is relative to alpha: at alpha 0.5 a pair at 0.5 (1 + 9e-5) is near."""
    q, k, v, blk, _ = _band_case(9e-5, alpha=0.5)
    assert oracle.block_select(q, k, 0, blk, 0.5, scale=1.0).near[0, 6, 0]
    q, k, v, blk, _ = _band_case(2e-4, alpha=0.5)
    assert not oracle.block_select(q, k, 0, blk, 0.5, scale=1.0).near.any()


def _sparse_row_by_hand(q, k, v, p, blk, kept_blocks, scale):
    """Row p of the block-sparse definition with math.exp loops (q: that row's query): exact
    keys j <= p of the kept blocks, one pooled term n_b exp(q . kbar_b * scale) vbar_b per
    skipped earlier block."""
    ob = p // blk
    terms = []
    for j in range(p + 1):
        if j // blk in kept_blocks:
            terms.append((sum(q[i] * k[j][i] for i in range(len(q))) * scale, 1.0, list(v[j])))
    for b in range(ob):
        if b not in kept_blocks:
            kb = [sum(k[j][i] for j in range(b * blk, (b + 1) * blk)) / blk for i in range(len(q))]
            vb = [sum(v[j][i] for j in range(b * blk, (b + 1) * blk)) / blk for i in range(len(q))]
            terms.append((sum(q[i] * kb[i] for i in range(len(q))) * scale, float(blk), vb))
    m = max(x for x, _, _ in terms)
    den = sum(n * math.exp(x - m) for x, n, _ in terms)
    return [sum(n * math.exp(x - m) * vv[i] for x, n, vv in terms) / den for i in range(len(q))]


def test_sparse_for_selection_follows_a_flipped_near_pair():
    """A selection that decides the near pair the other way gets the definition's output under
    that selection (checked against a hand-written row); the untouched rows keep the plain
    result; a selection that differs at a pair outside the band is refused."""
    q, k, v, blk, _ = _band_case(5e-5, t3=0.0, spread=1.5)
    base, sel = oracle.sparse(q, k, v, 0, blk, 0.1, scale=1.0)
    assert sel.kept[0, 6, 0, 1] and sel.kept[0, 7, 0, 1]
    flipped = sel.kept.copy()
    flipped[0, 6, 0, 1] = False                      # row 6 pools block 1 instead
    out, osel, rows = oracle.sparse_for_selection(q, k, v, 0, blk, 0.1, flipped, scale=1.0)
    assert rows.tolist() == [6]
    assert osel.near[0, 6, 0]
    want6 = _sparse_row_by_hand(q[0, 6, 0], k[0, :, 0], v[0, :, 0], 6, blk, {0, 3}, 1.0)
    want7 = _sparse_row_by_hand(q[0, 7, 0], k[0, :, 0], v[0, :, 0], 7, blk, {0, 1, 3}, 1.0)
    assert np.max(np.abs(out[0, 6, 0] - want6)) <= 1e-12
    assert np.max(np.abs(out[0, 7, 0] - want7)) <= 1e-12
    assert np.max(np.abs(out[0, 7, 0] - base[0, 7, 0])) <= 1e-15
    # the flip matters: pooling block 1 moves row 6 by several times the parity tolerance
    assert np.max(np.abs(out[0, 6, 0] - base[0, 6, 0])) > 4 * 5e-3
    bad = sel.kept.copy()
    bad[0, 6, 0, 2] = True                           # block 2 is far below the threshold
    with pytest.raises(ValueError, match="outside the threshold band"):
        oracle.sparse_for_selection(q, k, v, 0, blk, 0.1, bad, scale=1.0)
