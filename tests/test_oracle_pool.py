"""The process-pool harness of the long-prompt GPU parity test, checked on the CPU: fed the
oracle's own results it reports no error, and it catches a planted output error, a
selection that differs outside the threshold band, and follows a near pair decided the
other way."""
import numpy as np
import pytest

import oracle
import oracle_pool
import prefill_inputs as pi


def _pack(kept):
    """bool [R, H, nblk] -> uint32 words [R, H, W] (bit b % 32 of word b / 32)."""
    R, H, nblk = kept.shape
    W = (nblk + 31) // 32
    pad = np.zeros((R, H, W * 32), dtype=np.uint8)
    pad[..., :nblk] = kept
    return np.packbits(pad, axis=-1, bitorder="little").view(np.uint32)


@pytest.fixture(scope="module")
def case(tmp_path_factory):
    w = pi.planted_workload("pool-check", 31, 1, 4, 2, 64, 512, 256, "bf16")
    root = str(tmp_path_factory.mktemp("pool"))
    oracle_pool.save_inputs(w, root)
    return w, root


def _tasks(w, root, alpha=0.1, paths=("dense", "sparse")):
    return [oracle_pool.Task(root, w.dtype, p, s, w.chunk, g, w.Hq // w.Hkv, 128, alpha)
            for s in w.starts for g in range(w.Hkv) for p in paths]


def _write_oracle_results(w, root, alpha=0.1, edit=None):
    for s in w.starts:
        rows = np.arange(0, w.chunk, 3)
        q, kh, vh, kc, vc = (w.f64(x) for x in w.chunk_views(s))
        d = oracle.dense(q, kh, vh, kc, vc, s, rows=rows)[0].astype(np.float32)
        out, sel = oracle.sparse(q, w.f64(w.k[:, :s + w.chunk]), w.f64(w.v[:, :s + w.chunk]), s, 128, alpha,
                                 rows=rows)
        kept = sel.kept[0]
        out = out[0].astype(np.float32)
        if edit is not None:
            d, out, kept = edit(s, rows, d, out, kept, sel)
        oracle_pool.save_result(root, "dense", s, rows, d)
        oracle_pool.save_result(root, "sparse", s, rows, out, _pack(kept))


def test_pool_reports_no_error_on_the_oracles_own_results(case):
    w, root = case
    _write_oracle_results(w, root)
    summ = oracle_pool.summarize(oracle_pool.run_tasks(_tasks(w, root), workers=2))
    assert set(summ) == {(p, s) for p in ("dense", "sparse") for s in w.starts}
    for key, a in summ.items():
        assert a["finite"] and a["max"] <= 1e-6, (key, a)
        assert a["bad_pairs"] == 0 and a["rows_flipped"] == 0
    assert summ[("dense", 256)]["n"] == len(range(0, 256, 3)) * w.Hq * w.d


def test_pool_catches_planted_errors(case):
    w, root = case

    def edit(s, rows, d, out, kept, sel):
        if s == 256:
            d = d.copy()
            d[5, 3, 7] += 0.01
            kept = kept.copy()
            r = int(np.flatnonzero(rows >= 128)[0])            # a row with candidates
            far = np.flatnonzero(~kept[r, 0] & ~sel.near_pairs[0, r, 0] &
                                 (np.arange(kept.shape[-1]) < (s + rows[r]) // 128))
            kept[r, 0, far[0]] = True                          # keeps a block the definition skips
        return d, out, kept

    _write_oracle_results(w, root, edit=edit)
    summ = oracle_pool.summarize(oracle_pool.run_tasks(_tasks(w, root), workers=2))
    assert summ[("dense", 256)]["max"] >= 0.009
    assert summ[("dense", 0)]["max"] <= 1e-6
    assert summ[("sparse", 256)]["bad_pairs"] == 1
    assert summ[("sparse", 0)]["bad_pairs"] == 0


def test_pool_follows_a_near_pair_decided_the_other_way(case):
    """alpha is set to one candidate's own probability ratio, so that pair sits on the
    threshold (near); the stored selection drops it and the stored output is the definition's
    under that selection: no error, one flipped row."""
    w, root = case
    s = 256
    rows = np.arange(0, w.chunk, 3)
    q = w.f64(w.q[:, s:s + w.chunk])
    k = w.f64(w.k[:, :s + w.chunk])
    sel = oracle.block_select(q, k, s, 128, 0.1, rows=rows, heads=[0])
    r = int(np.flatnonzero(rows >= 200)[0])
    ob = (s + rows[r]) // 128
    sc = sel.scores[0, r, 0, :ob]
    ratio = np.exp(sc - sc.max())
    b = int(np.argsort(ratio)[-2])                   # the second-hottest candidate
    alpha = float(ratio[b])
    assert 0.0 < alpha < 1.0

    def edit(s_, rows_, d, out, kept, sel_):
        if s_ != s:
            return d, out, kept
        assert sel_.near_pairs[0, r, 0, b] and kept[r, 0, b]
        kept = kept.copy()
        kept[r, 0, b] = False
        ref, _, flipped = oracle.sparse_for_selection(
            q, k, w.f64(w.v[:, :s + w.chunk]), s, 128, alpha, kept[None], rows=rows_)
        assert r in flipped.tolist()
        return d, ref[0].astype(np.float32), kept

    _write_oracle_results(w, root, alpha=alpha, edit=edit)
    summ = oracle_pool.summarize(oracle_pool.run_tasks(_tasks(w, root, alpha, ("sparse",)), workers=2))
    a = summ[("sparse", s)]
    assert a["bad_pairs"] == 0 and a["rows_flipped"] >= 1 and a["near_rows"] >= 1
    assert a["max"] <= 1e-6
