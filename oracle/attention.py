"""Float64 CPU oracle for long-context prefill attention (dense and block-sparse).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything under ``oracle/``.  The CUDA library never calls it, and it shares no
code, header, table or helper with the CUDA path: its inputs are plain float64
numpy arrays (exact upcasts of the fp16/bf16 inputs).

Each function is the plain definition written out, row by row, with a numpy
matmul as the only library step: no tiling, no online softmax, no fusion.
Rows are computed in groups only to bound memory; every row's result depends
on that row alone.  The block-sparse function groups rows by their diagonal
block and takes a group's logits on the keys of the blocks some row of the
group keeps, a superset of each row's exact keys; every other key of a row is
masked to exp(-inf) = 0 exactly, so the grouping changes no row's value beyond
float64 summation order.

Sources (page title, section):
  * "Flash attention on ANE: fast long-context prefill", section
    "Flash attention: the core insight" -- softmax(Q K^T) V computed per query
    row; tiling is an implementation of the same result, so the oracle uses
    the untiled form.
  * "ANE Prefill Research", sections "How the ANE prefill path works" (a chunk
    of queries attends to a token-major K/V history plus its own keys, under
    an additive mask; the chunk's K/V are returned in cache layout) and
    "Folding a sparse indexer's selection into the mask" (dropped keys carry
    -30000, which exp() turns into an exact zero; the indexer's keep lists name
    compressed blocks of keys, and the keys after the last complete block stay
    visible).
  * "The Four Principles for Optimizing Transformers on the ANE", section
    "Masking in this layout" (masks are additive floats applied before the
    softmax).
  * "Porting FlashPrefill V2 to Apple silicon for faster prefill", sections
    "Compress keys before the heavy work" (mean-pool each key block),
    "A cheap map of where the attention lives" (one pooled score per query
    row per block; the local block stays exact), "The algorithm starts here"
    (keep blocks above alpha x the row's hottest block, plus the diagonal) and
    "Compute the peaks, summarize the rest" (kept blocks exact, skipped blocks
    represented by their pooled row).  The pooled correction weight is fixed
    by the benchmark spec: a skipped block b adds n_b * exp(q.kbar_b * scale)
    to the denominator and that weight times vbar_b to the numerator.

Readings where the pages are silent:
  * the mask is added after scaling: logits = (q.k) * scale + M;
  * mask=None means plain causal, the same as a 0 / -30000 causal mask;
  * with an explicit mask, visibility is the mask alone (it is arbitrary, not
    causal by contract), over all start_pos + C keys;
  * GQA: query head h reads KV head floor(h / (Hq / Hkv));
  * "above alpha x the hottest block" compares probabilities:
    exp(s_b - s_max) >= alpha; candidates are the strictly earlier blocks
    b < floor(p / block); the diagonal block floor(p / block) is always kept
    and never pooled; alpha = 0 keeps every candidate;
  * selection is per query row and per query head;
  * n_b is the number of keys in block b (the full block size for every
    candidate block, since candidates lie strictly before the query's block).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

MASK_DROP = -30000.0
_ROW_ELEMS = 1 << 24  # rows per group are sized so that a logits group is ~128 MB


def _rows_arg(rows, n):
    return np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)


def _heads_arg(heads, n):
    return list(range(n)) if heads is None else list(heads)


def causal_additive(C: int, start_pos: int, rows=None) -> np.ndarray:
    """0 where key j <= start_pos + i, else -30000; shape [len(rows), start_pos + C]."""
    rows = _rows_arg(rows, C)
    j = np.arange(start_pos + C)[None, :]
    return np.where(j <= start_pos + rows[:, None], 0.0, MASK_DROP)


# --------------------------------------------------------------------------
# dense chunked prefill
# --------------------------------------------------------------------------
def dense(q, k_hist, v_hist, k_chunk, v_chunk, start_pos, mask=None, scale=None, rows=None,
          heads=None, with_lse=False):
    """Attention of a chunk over [history ; chunk] keys.

    q [B, C, Hq, d]; k_hist, v_hist [B, s, Hkv, d]; k_chunk, v_chunk
    [B, C, Hkv, d]; mask [C, s + C] additive (shared by batch and heads) or
    None for causal.  For every row i (absolute position p = s + i) and head
    h: l_j = (q_i . k_j) * scale + M[i, j] over all keys j < s + C,
    o_i = sum_j exp(l_j - max l) v_j / sum_j exp(l_j - max l).
    Returns out [B, len(rows), len(heads), d]; with with_lse also
    lse [B, len(rows), len(heads)] = log sum_j exp(l_j), the log of the
    softmax denominator, which lets results over disjoint key sets be merged.
    """
    B, C, Hq, d = q.shape
    Hkv = k_chunk.shape[2]
    G = Hq // Hkv
    s = int(start_pos)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    k = np.concatenate([k_hist, k_chunk], axis=1)
    v = np.concatenate([v_hist, v_chunk], axis=1)
    T = s + C
    rows = _rows_arg(rows, C)
    heads = _heads_arg(heads, Hq)
    out = np.empty((B, len(rows), len(heads), d))
    lse = np.empty((B, len(rows), len(heads)))
    step = max(1, _ROW_ELEMS // T)
    jc = np.arange(C)[None, :]
    for b in range(B):
        for g in sorted({h // G for h in heads}):
            kg = np.ascontiguousarray(k[b, :, g, :])
            vg = np.ascontiguousarray(v[b, :, g, :])
            for hi, h in enumerate(heads):
                if h // G != g:
                    continue
                for r0 in range(0, len(rows), step):
                    rr = rows[r0:r0 + step]
                    logits = q[b, rr, h, :] @ kg.T
                    logits *= scale
                    if mask is None:
                        # causal: every history key (j < s) is visible; chunk key s + c gets
                        # -30000 where c > i (the columns below s would add 0)
                        logits[:, s:] += np.where(jc <= rr[:, None], 0.0, MASK_DROP)
                    else:
                        logits += mask[rr, :]
                    m = logits.max(axis=1, keepdims=True)
                    logits -= m
                    np.exp(logits, out=logits)
                    den = logits.sum(axis=1, keepdims=True)
                    out[b, r0:r0 + len(rr), hi, :] = (logits @ vg) / den
                    lse[b, r0:r0 + len(rr), hi] = m[:, 0] + np.log(den[:, 0])
    return (out, lse) if with_lse else out


def indexed_visible_keys(p: int, kept, ratio: int) -> np.ndarray:
    """The keys an indexer's compacted selection leaves visible to the query at position p.

    "ANE Prefill Research", section "Folding a sparse indexer's selection into the
    mask": the indexer keeps compressed blocks (keepIndices / keepCounts); block c
    covers keys ratio*c .. ratio*c + ratio - 1, and the keys after the last complete
    block, ratio*floor((p+1)/ratio) .. p, stay visible uncompressed (the pages' budget
    keptBlocks x compressRatio + (compressRatio - 1) counts them).  A kept block must
    be complete (c < floor((p+1)/ratio)); anything else is an error.  Returns the
    sorted distinct key indices.
    """
    if ratio < 1:
        raise ValueError("ratio %d < 1" % ratio)
    n_complete = (p + 1) // ratio
    kept = np.asarray(kept, dtype=np.int64).reshape(-1)
    if kept.size and (kept.min() < 0 or kept.max() >= n_complete):
        raise ValueError("kept block outside the %d complete blocks of position %d" % (n_complete, p))
    keys = (kept[:, None] * ratio + np.arange(ratio)[None, :]).reshape(-1)
    tail = np.arange(n_complete * ratio, p + 1)
    visible = np.unique(np.concatenate([keys, tail]))
    if visible.size == 0:
        raise ValueError("position %d sees no key" % p)
    return visible


def dense_indexed(q, k_hist, v_hist, k_chunk, v_chunk, start_pos, kept, ratio, scale=None,
                  rows=None, heads=None, with_lse=False):
    """Attention of a chunk over the keys an indexer kept, gathered per row.

    Row i (position p = start_pos + i) attends only to indexed_visible_keys(p,
    kept[i], ratio) of [history ; chunk]: o_i = sum_j exp(l_j - m) v_j / sum_j
    exp(l_j - m) over those keys j, l_j = (q_i . k_j) * scale.  The keys are
    gathered, no mask is formed; the pages state that folding the same selection
    into an additive mask as -30000 gives the same result, since exp() of such a
    logit is zero.  kept: a list of C index arrays.  Shapes and return as dense().
    """
    B, C, Hq, d = q.shape
    Hkv = k_chunk.shape[2]
    G = Hq // Hkv
    s = int(start_pos)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if len(kept) != C:
        raise ValueError("kept holds %d rows, expected %d" % (len(kept), C))
    k = np.concatenate([k_hist, k_chunk], axis=1)
    v = np.concatenate([v_hist, v_chunk], axis=1)
    rows = _rows_arg(rows, C)
    heads = _heads_arg(heads, Hq)
    out = np.empty((B, len(rows), len(heads), d))
    lse = np.empty((B, len(rows), len(heads)))
    for ri, i in enumerate(rows):
        js = indexed_visible_keys(s + int(i), kept[int(i)], ratio)
        for b in range(B):
            for hi, h in enumerate(heads):
                g = h // G
                logits = (k[b, js, g, :] @ q[b, i, h, :]) * scale
                m = logits.max()
                w = np.exp(logits - m)
                den = w.sum()
                out[b, ri, hi, :] = (w @ v[b, js, g, :]) / den
                lse[b, ri, hi] = m + math.log(den)
    return (out, lse) if with_lse else out


def chunk_kv_cache_layout(k_chunk):
    """The chunk's K (or V) in the head-major cache layout [B, Hkv, C, d]: a pure re-layout."""
    return np.ascontiguousarray(np.transpose(k_chunk, (0, 2, 1, 3)))


# --------------------------------------------------------------------------
# block-sparse prefill: pooled index
# --------------------------------------------------------------------------
def pool_blocks(x, block: int) -> np.ndarray:
    """Mean of each key block: x [B, T, H, d] -> [B, H, ceil(T / block), d]."""
    B, T, H, d = x.shape
    nblk = (T + block - 1) // block
    out = np.empty((B, H, nblk, d))
    for bk in range(nblk):
        out[:, :, bk, :] = x[:, bk * block:min(T, (bk + 1) * block)].mean(axis=1)
    return out


def block_counts(T: int, block: int) -> np.ndarray:
    nblk = (T + block - 1) // block
    return np.array([min(T, (bk + 1) * block) - bk * block for bk in range(nblk)], dtype=np.float64)


@dataclasses.dataclass
class Selection:
    kbar: np.ndarray      # [B, Hkv, nblk, d] pooled keys
    kept: np.ndarray      # bool [B, R, Hsel, nblk]: row keeps block (diagonal included)
    near: np.ndarray      # bool [B, R, Hsel]: row has a candidate within 1e-4 relative of alpha
    scores: np.ndarray    # [B, R, Hsel, nblk] pooled logits (q . kbar) * scale, all blocks
    rows: np.ndarray
    heads: list
    start_pos: int
    block: int
    # bool [B, R, Hsel, nblk]: the candidate's probability ratio exp(s_ib - s_max) lies within
    # 1e-4 relative of alpha, so float rounding may decide it either way (propagated through
    # the keep rules' group unions like ``near``); near = near_pairs.any(-1)
    near_pairs: np.ndarray = None


@dataclasses.dataclass(frozen=True)
class KeepRules:
    """Keep rules of the Metal port ("Porting FlashPrefill V2 to Apple silicon for faster
    prefill", the selection-map figure in "At 16k, only 28% of visible blocks run in
    full"): sinks, a local window and a dense tail are kept by rule; selection runs per
    32-position query tile; the map is per KV head.  Readings: a sink covers the blocks
    holding keys j < sink_tokens; the window is the local_blocks candidates just below
    the diagonal (the figure gives no width); the dense tail is the rows at positions
    p >= T - dense_tail_rows (T = start_pos + N, the end of the keys this call sees);
    a query tile's selection is the union of its rows' (each row keeps its own
    candidates only); a KV head's selection is the union of its query heads'."""
    sink_tokens: int = 0
    local_blocks: int = 0
    dense_tail_rows: int = 0
    row_group: int = 1
    share_kv_group: bool = False


def block_select(q, k, start_pos, block, alpha, scale=None, rows=None, heads=None,
                 near_rel=1e-4, rules=None) -> Selection:
    """Per-row block selection.

    q [B, N, Hq, d] (the chunk's queries), k [B, s + N, Hkv, d] (all keys).
    For row i at p = s + i: ob = floor(p / block); candidates b < ob;
    s_ib = (q_i . kbar_b) * scale; keep candidate b iff
    exp(s_ib - max_c s_ic) >= alpha; the diagonal block ob is always kept.
    rules (KeepRules): applied in order -- per-row rule keeps (sinks, window,
    dense tail), the union over aligned groups of row_group positions, the union
    over the query heads of a KV head; a group with a near row is near.
    """
    if rules is not None and (rules.row_group > 1 or rules.share_kv_group):
        return _select_grouped(q, k, start_pos, block, alpha, scale, rows, heads, near_rel, rules)
    B, N, Hq, d = q.shape
    T, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    s = int(start_pos)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kbar = pool_blocks(k, block)
    nblk = kbar.shape[2]
    rows = _rows_arg(rows, N)
    heads = _heads_arg(heads, Hq)
    ob = (s + rows) // block                                   # [R]
    cand = np.arange(nblk)[None, :] < ob[:, None]              # [R, nblk]
    kept = np.zeros((B, len(rows), len(heads), nblk), dtype=bool)
    near_pairs = np.zeros((B, len(rows), len(heads), nblk), dtype=bool)
    scores = np.empty((B, len(rows), len(heads), nblk))
    for b in range(B):
        for hi, h in enumerate(heads):
            sc = (q[b, rows, h, :] @ kbar[b, h // G].T) * scale   # [R, nblk]
            scores[b, :, hi] = sc
            smax = np.where(cand, sc, -np.inf).max(axis=1, keepdims=True)
            has = cand.any(axis=1)
            diff = np.where(cand, sc - np.where(has[:, None], smax, 0.0), -np.inf)
            ratio = np.exp(diff)                                      # p_b / p_max
            keep = cand & (ratio >= alpha)
            if rules is not None:
                bidx = np.arange(nblk)[None, :]
                keep |= cand & (bidx * block < rules.sink_tokens)
                keep |= cand & (bidx >= ob[:, None] - rules.local_blocks)
                keep |= cand & ((s + rows)[:, None] >= s + N - rules.dense_tail_rows)
            keep[np.arange(len(rows)), ob] = True
            kept[b, :, hi] = keep
            if alpha > 0:
                near_pairs[b, :, hi] = cand & (np.abs(ratio - alpha) <= near_rel * alpha)
    return Selection(kbar, kept, near_pairs.any(axis=-1), scores, rows, heads, s, block, near_pairs)


def _select_grouped(q, k, start_pos, block, alpha, scale, rows, heads, near_rel, rules):
    """block_select with the group unions: selects every row and head of the groups that
    the requested rows and heads belong to, takes the unions, returns the requested ones."""
    B, N, Hq, _ = q.shape
    G = Hq // k.shape[2]
    s = int(start_pos)
    rows = _rows_arg(rows, N)
    heads = _heads_arg(heads, Hq)
    g_rows = rules.row_group if rules.row_group > 1 else 1
    all_rows = np.arange(N)
    all_heads = list(range(Hq))
    base_rules = dataclasses.replace(rules, row_group=1, share_kv_group=False)
    full = block_select(q, k, s, block, alpha, scale, all_rows, all_heads, near_rel, base_rules)
    kept, near_pairs = full.kept.copy(), full.near_pairs.copy()
    ob = (s + all_rows) // block
    cand = np.arange(kept.shape[-1])[None, :] < ob[:, None]
    if g_rows > 1:
        grp = (s + all_rows) // g_rows
        for gi in np.unique(grp):
            m = grp == gi
            u = kept[:, m].any(axis=1, keepdims=True)              # [B, 1, Hq, nblk]
            kept[:, m] |= u & cand[m][None, :, None, :]
            near_pairs[:, m] |= near_pairs[:, m].any(axis=1, keepdims=True)
    if rules.share_kv_group:
        for g in range(Hq // G):
            hs = slice(g * G, (g + 1) * G)
            u = kept[:, :, hs].any(axis=2, keepdims=True)
            kept[:, :, hs] |= u
            near_pairs[:, :, hs] |= near_pairs[:, :, hs].any(axis=2, keepdims=True)
    hi = np.array(heads)
    np_sel = near_pairs[:, rows][:, :, hi]
    return Selection(full.kbar, kept[:, rows][:, :, hi], np_sel.any(axis=-1),
                     full.scores[:, rows][:, :, hi], rows, heads, s, block, np_sel)


def tile_union(kept_tile_rows) -> np.ndarray:
    """Sorted union of the kept blocks of a query tile's rows: kept_tile_rows bool [r, nblk]."""
    return np.flatnonzero(np.asarray(kept_tile_rows).any(axis=0)).astype(np.int32)


# --------------------------------------------------------------------------
# block-sparse prefill: exact kept blocks + pooled correction
# --------------------------------------------------------------------------
def sparse(q, k, v, start_pos, block, alpha, scale=None, rows=None, heads=None, sel=None,
           with_lse=False, rules=None):
    """Block-sparse attention with pooled correction.

    Row i (p = s + i), head h: kept set K_i from ``block_select``; skipped set
    R_i = {b < ob} minus K_i; exact keys E_i = {j <= p : floor(j / block) in K_i};
    with l_j = (q_i . k_j) * scale and s_ib the pooled logits,
      m = max(max_E l_j, max_R s_ib)
      o_i = (sum_E e^(l_j - m) v_j + sum_R n_b e^(s_ib - m) vbar_b)
            / (sum_E e^(l_j - m) + sum_R n_b e^(s_ib - m)).
    Returns (out [B, R, Hsel, d], sel); with with_lse also lse [B, R, Hsel], the
    log of the denominator above (exact and pooled terms).
    """
    B, N, Hq, d = q.shape
    T, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    s = int(start_pos)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if sel is None:
        sel = block_select(q, k, s, block, alpha, scale, rows, heads, rules=rules)
    rows, heads = sel.rows, sel.heads
    vbar = pool_blocks(v, block)
    nb = block_counts(T, block)
    nblk = len(nb)
    out = np.empty((B, len(rows), len(heads), d))
    lse = np.empty((B, len(rows), len(heads)))
    p_all = s + rows
    ob_all = p_all // block
    bidx = np.arange(nblk)[None, :]
    step = max(1, _ROW_ELEMS // T)
    for b in range(B):
        for g in sorted({h // G for h in heads}):
            kg = np.ascontiguousarray(k[b, :, g, :])
            vg = np.ascontiguousarray(v[b, :, g, :])
            his = [hi for hi, h in enumerate(heads) if h // G == g]
            # rows sharing a diagonal block share their candidates; a group's logits are taken
            # on the keys of the blocks some row of the group keeps for some head of this KV
            # head (a superset of every row's exact keys E_i), and each row masks the rest to
            # exp(-inf) = 0
            for obv in np.unique(ob_all):
                grp = np.flatnonzero(ob_all == obv)
                for r0 in range(0, len(grp), step):
                    sl = grp[r0:r0 + step]
                    rr, p = rows[sl], p_all[sl]
                    blocks = np.flatnonzero(sel.kept[b][sl][:, his].any(axis=(0, 1)))
                    if 2 * len(blocks) > nblk:
                        keys, ks, vs = np.arange(T), kg, vg
                    else:
                        keys = (blocks[:, None] * block + np.arange(block)[None, :]).reshape(-1)
                        keys = keys[keys < T]
                        ks, vs = kg[keys], vg[keys]
                    for hi in his:
                        h = heads[hi]
                        keep = sel.kept[b, sl, hi]                               # [r, nblk]
                        exact = keep[:, keys // block] & (keys[None, :] <= p[:, None])
                        skipped = (bidx < obv) & ~keep
                        logits = np.where(exact, (q[b, rr, h, :] @ ks.T) * scale, -np.inf)
                        pooled = np.where(skipped, sel.scores[b, sl, hi], -np.inf)
                        m = np.maximum(logits.max(axis=1), pooled.max(axis=1))[:, None]
                        we = np.exp(logits - m)
                        wp = nb[None, :] * np.exp(pooled - m)
                        num = we @ vs + wp @ vbar[b, g]
                        den = we.sum(axis=1) + wp.sum(axis=1)
                        out[b, sl, hi, :] = num / den[:, None]
                        lse[b, sl, hi] = m[:, 0] + np.log(den)
    return (out, sel, lse) if with_lse else (out, sel)


def skip_share(sel: Selection) -> float:
    """Share of off-diagonal candidate (row, block) pairs that were skipped."""
    ob = (sel.start_pos + sel.rows) // sel.block
    nblk = sel.kept.shape[-1]
    cand = np.arange(nblk)[None, :] < ob[:, None]                     # [R, nblk]
    n_cand = cand.sum() * sel.kept.shape[0] * sel.kept.shape[2]
    if n_cand == 0:
        return 0.0
    kept_cand = (sel.kept & cand[None, :, None, :]).sum()
    return float(1.0 - kept_cand / n_cand)


def sparse_for_selection(q, k, v, start_pos, block, alpha, kept, scale=None, rows=None, heads=None,
                         rules=None, with_lse=False):
    """Expected block-sparse output for a selection taken with finite-precision scores.

    A pair (row, block) whose probability ratio exp(s_ib - s_max) lies within 1e-4
    relative of alpha may be decided either way by rounding; any other pair is fixed
    by the definition (``block_select``).  ``kept`` (bool [B, R, Hsel, nblk]) must
    therefore equal the definition's selection outside those near pairs, else
    ValueError.  Returns (out, sel, flipped): out is the definition's output for each
    row under ``kept`` (rows that decided no near pair differently take the plain
    ``sparse`` result), sel the definition's selection, flipped the indices of the
    rows whose selection differs; with with_lse also the log of each row's
    denominator under ``kept``.
    """
    sel = block_select(q, k, start_pos, block, alpha, scale, rows, heads, rules=rules)
    kept = np.asarray(kept, dtype=bool)
    if kept.shape != sel.kept.shape:
        raise ValueError("kept has shape %s, expected %s" % (kept.shape, sel.kept.shape))
    diff = kept != sel.kept
    bad = diff & ~sel.near_pairs
    if bad.any():
        b, r, h, blk = (int(x[0]) for x in np.nonzero(bad))
        raise ValueError("selection differs from the definition at a pair outside the threshold band "
                         "(batch %d, row %d, head %d, block %d; %d such pairs)"
                         % (b, int(sel.rows[r]), sel.heads[h], blk, int(bad.sum())))
    out, _, lse = sparse(q, k, v, start_pos, block, alpha, scale, sel=sel, with_lse=True)
    flipped = np.flatnonzero(diff.any(axis=(0, 2, 3)))
    if flipped.size:
        alt = Selection(sel.kbar, kept[:, flipped], sel.near[:, flipped], sel.scores[:, flipped],
                        sel.rows[flipped], sel.heads, sel.start_pos, sel.block, sel.near_pairs[:, flipped])
        o_alt, _, l_alt = sparse(q, k, v, start_pos, block, alpha, scale, sel=alt, with_lse=True)
        out[:, flipped] = o_alt
        lse[:, flipped] = l_alt
    return (out, sel, flipped, lse) if with_lse else (out, sel, flipped)
