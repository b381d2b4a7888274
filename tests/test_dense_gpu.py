"""Dense chunked prefill: the CUDA path (through the C ABI) against the float64 oracle."""
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


def run_chunk(w, s, mask=None, out_kv=False, out_dtype=torch.float32):
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(s))
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    ok = ov = None
    if out_kv:
        B, C, Hkv, d = kc.shape
        ok = torch.empty((B, Hkv, C, d), dtype=kc.dtype, device="cuda")
        ov = torch.empty_like(ok)
    out = pfx.attn_dense(q, kh, vh, kc, vc, s, mask=dmask, out_k=ok, out_v=ov, out_dtype=out_dtype)
    pfx.stream_status()
    return out, ok, ov


def ref_chunk(w, s, mask=None, rows=None, heads=None):
    q, kh, vh, kc, vc = (w.f64(x) for x in w.chunk_views(s))
    return oracle.dense(q, kh, vh, kc, vc, s, mask=None if mask is None else mask.astype(np.float64),
                        rows=rows, heads=heads)


# --------------------------------------------------------------------------- config 1
@pytest.mark.parametrize("explicit", [True, False])
def test_config1_tiny_dense(explicit):
    w = pi.config(1)
    mask = pi.causal_mask(w.chunk, 0) if explicit else None
    out, _, _ = run_chunk(w, 0, mask)
    assert_close(out, ref_chunk(w, 0, mask), "config 1")


# --------------------------------------------------------------------------- config 2
@pytest.fixture(scope="module")
def cfg2():
    return pi.config(2)


@pytest.mark.parametrize("s", [0, 4096, 8192])
def test_config2_gqa_chunked_every_row(cfg2, s):
    """16q/8kv, d128, bf16, chunk 4096 at start 0/4096/8192 with the explicit causal mask."""
    w = cfg2
    mask = pi.causal_mask(w.chunk, s)
    out, ok, ov = run_chunk(w, s, mask, out_kv=True)
    assert_close(out, ref_chunk(w, s, mask), "config 2 s=%d" % s)
    _, _, _, kc, vc = w.chunk_views(s)
    assert np.array_equal(ok.cpu().view(torch.int16).numpy().view(np.uint16),
                          np.transpose(kc, (0, 2, 1, 3)))
    assert np.array_equal(ov.cpu().view(torch.int16).numpy().view(np.uint16),
                          np.transpose(vc, (0, 2, 1, 3)))


def test_config2_causal_default_matches_explicit_mask(cfg2):
    out_m, _, _ = run_chunk(cfg2, 4096, pi.causal_mask(cfg2.chunk, 4096))
    out_c, _, _ = run_chunk(cfg2, 4096, None)
    mx, _ = errors(out_c, out_m.double().cpu().numpy())
    assert mx <= 1e-3


# --------------------------------------------------------------------------- config 3
def test_config3_folded_indexer_mask():
    """Arbitrary mask: 512 compressed blocks of 4 per query over an 8192-token history."""
    w = pi.config(3)
    s = 8192
    mask, _ = pi.indexer_fold_mask(w.seed, w.chunk, s)
    out, _, _ = run_chunk(w, s, mask)
    ref = ref_chunk(w, s, mask)
    assert_close(out, ref, "config 3")
    # negative control: the causal-only arm must land >= 10x the tolerance away
    causal, _, _ = run_chunk(w, s, None)
    mx, _ = errors(causal, ref)
    assert mx >= 10 * MAX_ABS, mx


def test_config3_fp16_mask_matches():
    w = pi.config(3)
    s = 8192
    mask, _ = pi.indexer_fold_mask(w.seed, w.chunk, s)
    rows = sample_rows(w.chunk, 256, 3)
    out, _, _ = run_chunk(w, s, mask.astype(np.float16))
    assert_close(out[:, rows], ref_chunk(w, s, mask, rows=rows), "config 3 fp16 mask")


# --------------------------------------------------------------------------- edges
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 128), ("bf16", 64), ("f16", 64)])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 2), (3, 3)])
def test_ragged_chunks(dtype, d, Hq, Hkv):
    """Ragged chunk (C = 200, not a multiple of 128) over a 256-row history; GQA 2, 3 and 1."""
    w = pi.normal_workload("ragged", 11, 2, Hq, Hkv, d, 456, 200, dtype)
    for s in (0, 256):
        out, _, _ = run_chunk(w, s)
        assert_close(out, ref_chunk(w, s), "ragged s=%d" % s)


def test_ragged_explicit_mask_random_values():
    w = pi.normal_workload("ragged-mask", 12, 1, 4, 2, 128, 457, 201, "bf16")
    s = 256
    g = np.random.default_rng(5)
    mask = g.uniform(-4.0, 0.0, size=(w.chunk, s + w.chunk)).astype(np.float32)
    mask[g.random(mask.shape) < 0.5] = -30000.0
    mask[7, :] = -30000.0          # a fully masked row: plain softmax over the raw scores
    out, _, _ = run_chunk(w, s, mask)
    assert_close(out, ref_chunk(w, s, mask), "random mask")


def test_bf16_output_and_strided_query():
    w = pi.normal_workload("strided", 13, 1, 8, 4, 128, 640, 384, "bf16")
    s = 256
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(s))
    big = torch.zeros((1, 384, 12, 128), dtype=q.dtype, device="cuda")
    big[:, :, 2:10] = q
    qv = big[:, :, 2:10]                               # non-contiguous head slice
    out = pfx.attn_dense(qv, kh, vh, kc, vc, s, out_dtype=torch.bfloat16)
    pfx.stream_status()
    ref = ref_chunk(w, s)
    mx, _ = errors(out, ref)
    assert mx <= 5e-3 + 2 ** -8 * np.abs(ref).max()      # bf16 output adds half an ulp


def test_chunked_equals_one_shot_on_gpu():
    w = pi.normal_workload("oneshot", 14, 1, 8, 2, 128, 1024, 256, "bf16")
    q, k, v = dev(w.q, "bf16"), dev(w.k, "bf16"), dev(w.v, "bf16")
    one = pfx.attn_dense(q, k[:, :0], v[:, :0], k, v, 0)
    for s in range(0, 1024, 256):
        part = pfx.attn_dense(q[:, s:s + 256], k[:, :s], v[:, :s], k[:, s:s + 256], v[:, s:s + 256], s)
        mx, _ = errors(part, one[:, s:s + 256].double().cpu().numpy())
        assert mx <= 2e-3
    pfx.stream_status()


def test_cache_copy_batch_ragged_strided():
    """The chunk's K/V copied into a larger head-major cache: batch 2, 3 KV heads, head dim 64,
    a ragged 200-row chunk written at rows 256..455 of a 512-row cache.  A bit copy; the cache
    rows outside the chunk keep their sentinel values."""
    w = pi.normal_workload("cache-copy", 15, 2, 6, 3, 64, 456, 200, "bf16")
    s, C = 256, 200
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(s))
    ck = torch.full((2, 3, 512, 64), -7.0, dtype=torch.bfloat16, device="cuda")
    cv = torch.full_like(ck, 5.0)
    pfx.attn_dense(q, kh, vh, kc, vc, s, out_k=ck[:, :, s:s + C], out_v=cv[:, :, s:s + C])
    pfx.stream_status()
    _, _, _, kcn, vcn = w.chunk_views(s)
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits(ck[:, :, s:s + C]), np.transpose(kcn, (0, 2, 1, 3)))
    assert np.array_equal(bits(cv[:, :, s:s + C]), np.transpose(vcn, (0, 2, 1, 3)))
    assert bool((ck[:, :, :s] == -7.0).all()) and bool((ck[:, :, s + C:] == -7.0).all())
    assert bool((cv[:, :, :s] == 5.0).all()) and bool((cv[:, :, s + C:] == 5.0).all())


def test_launch_counter_counts_kernels():
    w = pi.config(1)
    pfx.launch_count(reset=True)
    run_chunk(w, 0, None, out_kv=True)
    assert pfx.launch_count() == 2      # attention + one cache-layout copy of K and V
    pfx.launch_count(reset=True)
    run_chunk(w, 0, pi.causal_mask(w.chunk, 0))
    assert pfx.launch_count() == 3      # mask packing, the bits launch, the values launch


def test_value_outside_fp16_range_is_reported():
    """P * V runs in fp16; a bf16 v beyond +-65504 must be refused loudly, not rounded to inf."""
    w = pi.normal_workload("vrange", 15, 1, 4, 2, 128, 256, 256, "bf16")
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(0))
    vc[0, 17, 1, 5] = 1.0e6
    pfx.attn_dense(q, kh, vh, kc, vc, 0)
    with pytest.raises(pfx.PFError) as e:
        pfx.stream_status()
    assert e.value.status == pf.PF_ERANGE
    vc[0, 17, 1, 5] = float("nan")
    pfx.attn_dense(q, kh, vh, kc, vc, 0)
    with pytest.raises(pfx.PFError) as e:
        pfx.stream_status()
    assert e.value.status == pf.PF_ERANGE
    vc[0, 17, 1, 5] = 1.0
    pfx.attn_dense(q, kh, vh, kc, vc, 0)
    pfx.stream_status()


# --------------------------------------------------------------------------- tail split
@pytest.mark.parametrize("case", ["causal", "mask", "ragged", "bf16-out"])
def test_tail_split_matches_oracle_and_unsplit(case):
    """32 units (8 query tiles x 4 head pairs) on a 152-SM GPU: with a workspace every unit's
    key range is cut into parts whose partial (O, m, l) are merged on the device; the result
    must meet the oracle like the unsplit call does."""
    C = 1000 if case == "ragged" else 1024
    w = pi.normal_workload("split-" + case, 61, 1, 8, 2, 128, 2048 + C, C, "bf16")
    s = 2048
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(s))
    mask = None
    if case == "mask":
        g = np.random.default_rng(62)
        mask = np.zeros((C, s + C), dtype=np.float32)
        mask[g.random(mask.shape) < 0.3] = -30000.0
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    odt = torch.bfloat16 if case == "bf16-out" else torch.float32
    split = pfx.attn_dense(q, kh, vh, kc, vc, s, mask=dmask, out_dtype=odt, workspace=True)
    whole = pfx.attn_dense(q, kh, vh, kc, vc, s, mask=dmask, out_dtype=odt, workspace=None)
    pfx.stream_status()
    ref = ref_chunk(w, s, mask)
    if case == "bf16-out":
        for out in (split, whole):
            mx, _ = errors(out, ref)
            assert mx <= 5e-3 + 2 ** -8 * np.abs(ref).max()
    else:
        assert_close(split, ref, "split " + case)
        assert_close(whole, ref, "whole " + case)
    mx, _ = errors(split, whole.double().cpu().numpy())
    assert mx <= 2e-3


def _tile_sparse_mask(seed, C, T, keep_tiles):
    """Binary mask where query tile i keeps keep_tiles[i] random key tiles (each key of those
    kept with probability 0.6) and drops every other key; every row keeps at least one key."""
    g = np.random.default_rng(seed)
    nkt = -(-T // 128)
    mask = np.full((C, T), -30000.0, dtype=np.float32)
    for qt, n in enumerate(keep_tiles):
        r0, r1 = qt * 128, min(C, qt * 128 + 128)
        tiles = g.choice(nkt, n, replace=False)
        for t in tiles:
            blk = mask[r0:r1, t * 128:min(T, t * 128 + 128)]
            blk[g.random(blk.shape) < 0.6] = 0.0
        mask[r0:r1, tiles[0] * 128] = 0.0
    return mask


@pytest.mark.parametrize("workspace", [True, None])
def test_binary_mask_skips_dropped_key_tiles(workspace):
    """A binary mask that drops whole 128-key tiles for a query tile: with the workspace the
    packed path visits only the kept tiles (query tiles keeping 1 or 2 of 24 tiles leave tail
    split parts with no tile at all); without it every tile is read through the mask values.
    Both against the oracle."""
    C, s = 1000, 2048
    w = pi.normal_workload("tile-skip", 81, 1, 8, 2, 128, s + C, C, "bf16")
    mask = _tile_sparse_mask(82, C, s + C, [1, 2, 3, 5, 24, 8, 1, 13])
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(s))
    lse = torch.empty((1, 8, C), dtype=torch.float32, device="cuda")
    out = pfx.attn_dense(q, kh, vh, kc, vc, s, mask=torch.from_numpy(mask).cuda(), lse=lse,
                         workspace=workspace)
    pfx.stream_status()
    ref, rlse = oracle.dense(*(w.f64(x) for x in w.chunk_views(s)), s, mask=mask.astype(np.float64),
                             with_lse=True)
    assert_close(out, ref, "tile-sparse mask, workspace %s" % workspace)
    got = lse.cpu().double().numpy().transpose(0, 2, 1)
    assert np.max(np.abs(got - rlse)) <= LSE_TOL


def test_binary_mask_past_the_tile_bitmap_visits_every_tile():
    """start_pos + C = 262272 keys is 2050 key tiles, more than a query tile's 2048-bit bitmap:
    the packed bits are still used but every key tile is visited.  Sampled rows."""
    C, s = 200, 262144
    w = pi.normal_workload("tile-bitmap-cap", 83, 1, 2, 1, 128, s + C, C, "bf16")
    mask = _tile_sparse_mask(84, C, s + C, [40, 3])
    rows = np.array([0, 1, 63, 127, 128, 150, 199])
    out, _, _ = run_chunk(w, s, mask)
    ref = ref_chunk(w, s, mask, rows=rows)
    assert_close(out[:, rows], ref, "2050 key tiles")


@pytest.mark.parametrize("kind", ["binary", "values"])
def test_mask_broadcast_over_batch(kind):
    """A [C, s + C] mask applies to every batch and head: batch 2, a ragged chunk over a
    history, the mask read as bits with dropped key tiles skipped (binary) or as values."""
    C, s = 300, 256
    w = pi.normal_workload("mask-batch", 87, 2, 4, 2, 128, s + C, C, "bf16")
    if kind == "binary":
        mask = _tile_sparse_mask(88, C, s + C, [2, 3, 5])
    else:
        g = np.random.default_rng(89)
        mask = np.where(g.random((C, s + C)) < 0.3, -30000.0, g.normal(0.0, 2.0, (C, s + C))).astype(np.float32)
    out, _, _ = run_chunk(w, s, mask)
    assert_close(out, ref_chunk(w, s, mask), "batch 2, %s mask" % kind)


def test_binary_mask_tile_bitmap_above_1024_tiles():
    """start_pos + C = 150088 keys is 1173 key tiles (the last one 72 keys long): a query tile's
    bitmap spans 37 words, and the kept tiles past tile 1024 land in the packing pass's second
    per-lane bitmap word.  Query tile 0 keeps tiles 3, 1100 and the ragged last one, query tile 1
    keeps tiles 500 and 1050; a bit lost from the bitmap drops a kept tile.  Sampled rows of both
    query tiles against the oracle."""
    C, s = 200, 149888
    T = s + C
    w = pi.normal_workload("tile-bitmap-hi", 85, 1, 2, 1, 128, T, C, "bf16")
    g = np.random.default_rng(86)
    mask = np.full((C, T), -30000.0, dtype=np.float32)
    for (r0, r1), kept in (((0, 128), (3, 1100, 1172)), ((128, C), (500, 1050))):
        for t in kept:
            blk = mask[r0:r1, t * 128:min(T, t * 128 + 128)]
            blk[g.random(blk.shape) < 0.6] = 0.0
        mask[r0:r1, kept[1] * 128] = 0.0
    rows = np.array([0, 5, 77, 127, 128, 160, 199])
    out, _, _ = run_chunk(w, s, mask)
    ref = ref_chunk(w, s, mask, rows=rows)
    assert_close(out[:, rows], ref, "1173 key tiles")


@pytest.mark.parametrize("mdtype", [np.float32, np.float16])
@pytest.mark.parametrize("tail", [0.0, -30000.0, -2.0])
@pytest.mark.parametrize("padded", [True, False])
def test_padded_mask_rows_with_ragged_keys(mdtype, tail, padded):
    """start_pos + C = 941 keys per mask row, not a multiple of 4.  Rows padded to a 16-byte
    stride: the packing pass reads them with vector loads and the last key of each row on its
    own; contiguous rows (941 values apart, not on 16-byte boundaries): the scalar packing pass.
    The rows' last key carries `tail` in every third row (kept, dropped, or a non-binary value
    that sends the call to the value path); the padding holds NaN, which no row may read."""
    C, s = 301, 640
    T = s + C
    ld = (T + 7) // 8 * 8 + 8 if padded else T
    w = pi.normal_workload("padded-mask", 91, 1, 4, 2, 128, T, C, "bf16")
    g = np.random.default_rng(92)
    vals = np.where(g.random((C, T)) < 0.4, -30000.0, 0.0)
    vals[:, 0] = 0.0
    vals[::3, T - 1] = tail
    full = np.full((C, ld), np.nan)
    full[:, :T] = vals
    dmask = torch.from_numpy(full.astype(mdtype)).cuda()[:, :T]
    assert dmask.stride(0) == ld
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(s))
    out = pfx.attn_dense(q, kh, vh, kc, vc, s, mask=dmask)
    pfx.stream_status()
    assert_close(out, ref_chunk(w, s, vals.astype(mdtype)), "padded mask rows, tail %g" % tail)


def test_tail_split_workspace_too_small_is_refused():
    w = pi.normal_workload("split-small-ws", 63, 1, 8, 2, 128, 1024, 512, "bf16")
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(512))
    with pytest.raises(pfx.PFError) as e:
        pfx.attn_dense(q, kh, vh, kc, vc, 512, workspace=torch.empty(1024, dtype=torch.uint8, device="cuda"))
    assert e.value.status == pf.PF_EINVAL


# --------------------------------------------------------------------------- log-sum-exp
LSE_TOL = 1e-4   # fp32 scores and sums, ex2/lg2 approximations: ~1e-6 relative on |lse| ~ 10


@pytest.mark.parametrize("case", ["causal", "mask", "split"])
def test_lse_matches_oracle(case):
    C, s = 1024, 2048
    w = pi.normal_workload("lse-" + case, 71, 1, 8, 2, 128, s + C, C, "bf16")
    q, kh, vh, kc, vc = (dev(x, w.dtype) for x in w.chunk_views(s))
    mask = None
    if case == "mask":
        mask = np.zeros((C, s + C), dtype=np.float32)
        mask[np.random.default_rng(72).random(mask.shape) < 0.3] = -30000.0
    lse = torch.empty((1, 8, C), dtype=torch.float32, device="cuda")
    out = pfx.attn_dense(q, kh, vh, kc, vc, s, mask=None if mask is None else torch.from_numpy(mask).cuda(),
                         lse=lse, workspace=True if case == "split" else None)
    pfx.stream_status()
    ref, rlse = oracle.dense(*(w.f64(x) for x in w.chunk_views(s)), s,
                             mask=None if mask is None else mask.astype(np.float64), with_lse=True)
    assert_close(out, ref, "lse case " + case)
    got = lse.cpu().double().numpy().transpose(0, 2, 1)          # [B, C, Hq]
    assert np.max(np.abs(got - rlse)) <= LSE_TOL, np.max(np.abs(got - rlse))


# --------------------------------------------------------------------------- the bench's launches
@pytest.mark.slow
def test_config4_dense_chunked_as_benchmarked(tmp_path):
    """The 32K prompt as bench.py runs it: 8 chunks of 4096 causal rows over the previous
    chunks' K/V, chunk outputs written into one [1, 32768, 32, 128] tensor, K/V emitted into a
    head-major cache, the tail-split workspace on, v kept in fp16 (each chunk's v converted once).
    Per chunk 2048 seeded rows, the last 128 rows and every tile-boundary row, all 32 heads, against
    the oracle (a process pool, one task per chunk and KV head); the cache must be a bit copy of
    k and of the fp16 v."""
    import oracle_pool
    w = pi.config(4)
    N, CH = w.N, 4096
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    Q, K, V = to(w.q), to(w.k), to(w.v)
    out = torch.empty((1, N, 32, 128), dtype=torch.float32, device="cuda")
    ck = torch.empty((1, 8, N, 128), dtype=torch.bfloat16, device="cuda")
    cv = torch.empty((1, 8, N, 128), dtype=torch.float16, device="cuda")
    V16 = torch.empty(V.shape, dtype=torch.float16, device="cuda")
    for s in range(0, N, CH):
        pfx.to_f16(V[:, s:s + CH], out=V16[:, s:s + CH])
        pfx.attn_dense(Q[:, s:s + CH], K[:, :s], V16[:, :s], K[:, s:s + CH], V16[:, s:s + CH], s,
                       out=out[:, s:s + CH], out_k=ck[:, :, s:s + CH], out_v=cv[:, :, s:s + CH])
    pfx.stream_status()
    assert torch.equal(ck.transpose(1, 2).contiguous(), K)
    assert torch.equal(cv.transpose(1, 2).contiguous(), V16)  # the cache holds the fp16 v bit for bit
    root = str(tmp_path)
    oracle_pool.save_inputs(w, root)
    tasks = []
    for ci, s in enumerate(range(0, N, CH)):
        rows = sample_rows(CH, 2048, 400 + ci)
        oracle_pool.save_result(root, "dense", s, rows, out[0, s + torch.from_numpy(rows).cuda()].cpu().numpy())
        tasks += [oracle_pool.Task(root, w.dtype, "dense", s, CH, g, w.Hq // w.Hkv) for g in range(w.Hkv)]
    for (path, s), a in sorted(oracle_pool.summarize(oracle_pool.run_tasks(tasks)).items()):
        assert a["finite"] and a["n"] >= 2048 * 32 * 128, (s, a)
        assert a["max"] <= MAX_ABS and a["mean"] <= MEAN_ABS, ("32K chunk at %d" % s, a["max"], a["mean"])
