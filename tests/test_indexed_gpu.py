"""Index-driven attention (pf_attn_indexed): the CUDA path against the float64 oracle's gathered
form, and against the explicit-mask path with the same selection folded into a -30000 mask."""
import numpy as np
import pytest
import torch

import oracle
import prefill_inputs as pi
from gpu_util import assert_close, dev, errors, sample_rows
from long_context_prefill_chunked_gb300 import pf

pytestmark = pytest.mark.gpu

pfx = pytest.importorskip("long_context_prefill_chunked_gb300")

LSE_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    pfx.set_wait_timeout(400_000_000)
    yield
    pfx.stream_status()


def keep_tensors(kept, stride=None):
    """Ragged per-row keep lists -> int32 keep_idx [C, stride] (padded with -7, never read) and
    keep_cnt [C] on the device."""
    C = len(kept)
    stride = max(1, max(len(k) for k in kept)) if stride is None else stride
    idx = np.full((C, stride), -7, dtype=np.int32)
    cnt = np.zeros(C, dtype=np.int32)
    for i, k in enumerate(kept):
        idx[i, :len(k)] = k
        cnt[i] = len(k)
    return torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()


def views(w, s):
    return [dev(x, w.dtype) for x in w.chunk_views(s)]


def test_config3_selection_matches_oracle_and_folded_mask():
    """Config 3's 512 compressed blocks of 4 per query over an 8192-token history: given as keep
    lists it must equal the oracle's gathered attention, and bit for bit the explicit-mask path
    fed the same selection folded into a mask (both read the same bits)."""
    w = pi.config(3)
    s = 8192
    mask, kept = pi.indexer_fold_mask(w.seed, w.chunk, s)
    q, kh, vh, kc, vc = views(w, s)
    idx, cnt = keep_tensors(kept)
    lse = torch.empty((1, w.Hq, w.chunk), dtype=torch.float32, device="cuda")
    out = pfx.attn_indexed(q, kh, vh, kc, vc, s, idx, cnt, 4, lse=lse)
    folded = pfx.attn_dense(q, kh, vh, kc, vc, s, mask=torch.from_numpy(mask).cuda())
    pfx.stream_status()
    assert torch.equal(out, folded)
    rows = sample_rows(w.chunk, 256, 31)
    ref, rlse = oracle.dense_indexed(*(w.f64(x) for x in w.chunk_views(s)), s, kept, 4, rows=rows,
                                     with_lse=True)
    assert_close(out[:, rows], ref, "config 3 keep lists")
    got = lse.cpu().double().numpy().transpose(0, 2, 1)[:, rows]
    assert np.max(np.abs(got - rlse)) <= LSE_TOL


@pytest.mark.parametrize("ratio,dtype,d,Hq,Hkv", [(3, "bf16", 128, 4, 2), (5, "f16", 64, 2, 2),
                                                 (1, "bf16", 128, 6, 2)])
def test_ragged_lists_every_row(ratio, dtype, d, Hq, Hkv):
    """Ragged chunk (333 rows at 256), lists of varying length with repeats and any order, a
    keep_stride past the longest list; every row against the oracle, with the log-sum-exp."""
    C, s = 333, 256
    w = pi.normal_workload("indexed-%d" % ratio, 90 + ratio, 1, Hq, Hkv, d, s + C, C, dtype)
    g = np.random.default_rng(91 + ratio)
    kept = []
    for i in range(C):
        nc = (s + i + 1) // ratio
        k = g.choice(nc, size=int(g.integers(1, min(nc, 40) + 1)), replace=False)
        if len(k) > 2:
            k = np.concatenate([k, k[:2]])           # repeats count once
        kept.append(g.permutation(k))
    idx, cnt = keep_tensors(kept, stride=48)
    q, kh, vh, kc, vc = views(w, s)
    lse = torch.empty((1, Hq, C), dtype=torch.float32, device="cuda")
    out = pfx.attn_indexed(q, kh, vh, kc, vc, s, idx, cnt, ratio, lse=lse)
    pfx.stream_status()
    ref, rlse = oracle.dense_indexed(*(w.f64(x) for x in w.chunk_views(s)), s, kept, ratio, with_lse=True)
    assert_close(out, ref, "ratio %d" % ratio)
    got = lse.cpu().double().numpy().transpose(0, 2, 1)
    assert np.max(np.abs(got - rlse)) <= LSE_TOL


def test_lists_in_few_key_tiles_with_the_tail_split():
    """32 units on 152 SMs (the tail split cuts every unit into parts); each query tile keeps
    blocks from two or three 128-key tiles only, so most parts of a unit visit no tile."""
    C, s, ratio = 1024, 2048, 4
    w = pi.normal_workload("indexed-split", 93, 1, 8, 2, 128, s + C, C, "bf16")
    g = np.random.default_rng(94)
    kept = []
    for qt in range(C // 128):
        hi = (s + qt * 128 + 1) // 128                 # key tiles complete for every row of the tile
        tiles = g.choice(hi, size=min(hi, 2 + qt % 2), replace=False)
        blocks = np.concatenate([np.arange(t * 32, t * 32 + 32) for t in tiles])
        for r in range(128):
            kept.append(g.choice(blocks, size=12, replace=False))
    idx, cnt = keep_tensors(kept)
    q, kh, vh, kc, vc = views(w, s)
    split = pfx.attn_indexed(q, kh, vh, kc, vc, s, idx, cnt, ratio)
    pfx.stream_status()
    ref = oracle.dense_indexed(*(w.f64(x) for x in w.chunk_views(s)), s, kept, ratio)
    assert_close(split, ref, "indexed, split parts")


def test_invalid_selection_is_reported():
    """An entry naming an incomplete block, a count past keep_stride, or a row that sees no key
    cannot be checked on the host: the packing pass skips it and the stream status reports
    PF_EINVAL; the next valid call is unaffected."""
    C, s, ratio = 128, 128, 4
    w = pi.normal_workload("indexed-bad", 95, 1, 2, 2, 128, s + C, C, "bf16")
    q, kh, vh, kc, vc = views(w, s)
    good = [np.array([0, 5]) for _ in range(C)]
    for bad_rows in (
        {3: np.array([(s + 3 + 1) // ratio])},          # the block ending past row 3
        {7: np.array([-1])},
        {9: np.array([1 << 30])},
    ):
        kept = [bad_rows.get(i, good[i]) for i in range(C)]
        idx, cnt = keep_tensors(kept)
        pfx.attn_indexed(q, kh, vh, kc, vc, s, idx, cnt, ratio)
        with pytest.raises(pfx.PFError) as e:
            pfx.stream_status()
        assert e.value.status == pf.PF_EINVAL
    idx, cnt = keep_tensors(good, stride=2)
    cnt[5] = 3                                          # past keep_stride
    pfx.attn_indexed(q, kh, vh, kc, vc, s, idx, cnt, ratio)
    with pytest.raises(pfx.PFError) as e:
        pfx.stream_status()
    assert e.value.status == pf.PF_EINVAL
    # row i = 3 sits at p = 131: (p + 1) % 4 == 0, so with an empty list it sees no key
    kept = [np.array([], dtype=np.int64) if i == 3 else good[i] for i in range(C)]
    idx, cnt = keep_tensors(kept)
    pfx.attn_indexed(q, kh, vh, kc, vc, s, idx, cnt, ratio)
    with pytest.raises(pfx.PFError) as e:
        pfx.stream_status()
    assert e.value.status == pf.PF_EINVAL
    idx, cnt = keep_tensors(good)
    out = pfx.attn_indexed(q, kh, vh, kc, vc, s, idx, cnt, ratio)
    pfx.stream_status()
    ref = oracle.dense_indexed(*(w.f64(x) for x in w.chunk_views(s)), s, good, ratio)
    assert_close(out, ref, "valid call after invalid ones")
