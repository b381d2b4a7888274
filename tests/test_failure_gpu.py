"""Failure detection without a GPU fault: a withheld completion signal makes the
kernels' bounded waits run out; the host reads PF_ETIMEOUT from the device status
word and the context stays usable."""
import numpy as np
import pytest

import oracle
import prefill_inputs as pi
from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

pfx = pytest.importorskip("long_context_prefill_chunked_gb300")
from long_context_prefill_chunked_gb300 import pf  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    pfx.set_debug_withhold(False)
    pfx.set_wait_timeout(400_000_000)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_withheld_signal_times_out_and_context_survives(dtype):
    w = pi.normal_workload("withhold", 41, 1, 4, 2, 128, 512, 256, dtype)
    s = 256
    q, kh, vh, kc, vc = (dev(x, dtype) for x in w.chunk_views(s))
    pfx.stream_status()
    pfx.set_wait_timeout(20_000_000)          # ~10 ms: nothing legitimate waits that long
    pfx.set_debug_withhold(True)
    try:
        pfx.attn_dense(q, kh, vh, kc, vc, s)
        with pytest.raises(pfx.PFError) as e:
            pfx.stream_status()
        assert e.value.status == pf.PF_ETIMEOUT
    finally:
        pfx.set_debug_withhold(False)
        pfx.set_wait_timeout(400_000_000)
    out = pfx.attn_dense(q, kh, vh, kc, vc, s)
    pfx.stream_status()
    ref = oracle.dense(*(w.f64(x) for x in w.chunk_views(s)), s)
    assert_close(out, ref, "after a timeout")


def test_withheld_signal_times_out_in_block_sparse_attention():
    """The same for the block-sparse attention: its kernel gives up on the withheld S tile,
    reports PF_ETIMEOUT, and the next call over the same selection is correct."""
    w = pi.planted_workload("withhold-sparse", 42, 1, 4, 2, 128, 1024, 1024, "bf16")
    q, k, v = (dev(x, w.dtype) for x in (w.q, w.k, w.v))
    sel = pfx.block_index(q, k, 0, 128, 0.1)
    pfx.stream_status()
    pfx.set_wait_timeout(20_000_000)
    pfx.set_debug_withhold(True)
    try:
        pfx.attn_sparse(q, k, v, 0, sel)
        with pytest.raises(pfx.PFError) as e:
            pfx.stream_status()
        assert e.value.status == pf.PF_ETIMEOUT
    finally:
        pfx.set_debug_withhold(False)
        pfx.set_wait_timeout(400_000_000)
    out = pfx.attn_sparse(q, k, v, 0, sel)
    pfx.stream_status()
    words = sel.row_bits.cpu().numpy().view(np.uint32)
    bits = np.unpackbits(words.view(np.uint8).reshape(*words.shape, 4), axis=-1, bitorder="little")
    kept = np.transpose(bits.reshape(*words.shape[:3], -1)[..., :8].astype(bool), (0, 2, 1, 3))
    ref, _, _ = oracle.sparse_for_selection(w.f64(w.q), w.f64(w.k), w.f64(w.v), 0, 128, 0.1, kept)
    assert_close(out, ref, "sparse after a timeout")
