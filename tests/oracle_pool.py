"""The float64 oracle over a whole chunked prompt, one (chunk, KV head) task per worker.

Test infrastructure.  A GPU parity test runs every chunk of a long prompt on the
GPU, stores the sampled rows' outputs and selections next to the prompt's input
bits in a scratch directory, and hands this module one task per (chunk, KV head).
Each task runs in a spawned worker process (one BLAS thread each, so the workers
fill the host's cores without oversubscribing them), computes the oracle's dense
and block-sparse results for its rows and the KV head's query heads, and returns
error statistics only.

Block-sparse rows: the GPU's row selection must equal the oracle's except at
near-threshold (row, block) pairs, whose probability ratio lies within 1e-4
relative of alpha so that rounding may decide them either way.  Every row's
output is compared: where the GPU decided a near pair the other way, the expected
output is the oracle's output under the oracle's selection with exactly those
near pairs flipped, which is itself a valid selection.
"""
from __future__ import annotations

import dataclasses
import multiprocessing as mp
import os

import numpy as np

_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def unpack_words(words: np.ndarray, nblk: int) -> np.ndarray:
    """uint32 [..., W] (bit b % 32 of word b / 32) -> bool [..., nblk]."""
    w = np.ascontiguousarray(words).view(np.uint32)
    bits = np.unpackbits(w.view(np.uint8).reshape(*w.shape, 4), axis=-1, bitorder="little")
    return bits.reshape(*w.shape[:-1], -1)[..., :nblk].astype(bool)


def save_inputs(w, root: str) -> None:
    """The prompt's input bits, memory-mapped by the workers."""
    for name in ("q", "k", "v"):
        np.save(os.path.join(root, name + ".npy"), getattr(w, name))


def save_result(root: str, path: str, s: int, rows, out=None, row_words=None) -> None:
    """One chunk's GPU result on the sampled rows: out [R, Hq, d] float32 and, for the sparse
    path, the row selection words [R, Hq, W] uint32."""
    np.save(os.path.join(root, "%s_%d_rows.npy" % (path, s)), np.asarray(rows, dtype=np.int64))
    if out is not None:
        np.save(os.path.join(root, "%s_%d_out.npy" % (path, s)), out)
    if row_words is not None:
        np.save(os.path.join(root, "%s_%d_bits.npy" % (path, s)), row_words)


@dataclasses.dataclass
class Task:
    root: str
    dtype: str
    path: str          # "dense" or "sparse"
    s: int             # chunk start
    C: int             # chunk rows
    g: int             # KV head
    G: int             # query heads per KV head
    block: int = 128
    alpha: float = 0.1


def _err_stats(gpu: np.ndarray, ref: np.ndarray) -> dict:
    e = np.abs(gpu.astype(np.float64) - ref)
    return {"n": int(e.size), "sum": float(e.sum()), "max": float(e.max()) if e.size else 0.0,
            "finite": bool(np.isfinite(gpu).all())}


def run_task(t: Task) -> dict:
    import oracle
    import prefill_inputs as pi

    def load(name):
        return np.load(os.path.join(t.root, name), mmap_mode="r")

    rows = load("%s_%d_rows.npy" % (t.path, t.s))
    hs = slice(t.g * t.G, (t.g + 1) * t.G)
    T = t.s + t.C
    q = pi.bits_to_f64(np.ascontiguousarray(load("q.npy")[:, t.s:T, hs]), t.dtype)        # [B, C, G, d]
    k = pi.bits_to_f64(np.ascontiguousarray(load("k.npy")[:, :T, t.g:t.g + 1]), t.dtype)  # [B, T, 1, d]
    v = pi.bits_to_f64(np.ascontiguousarray(load("v.npy")[:, :T, t.g:t.g + 1]), t.dtype)
    gpu = np.asarray(load("%s_%d_out.npy" % (t.path, t.s))[:, hs])                        # [R, G, d]
    res = {"path": t.path, "s": t.s, "g": t.g}
    if t.path == "dense":
        ref = oracle.dense(q, k[:, :t.s], v[:, :t.s], k[:, t.s:], v[:, t.s:], t.s, rows=rows)
        res.update(_err_stats(gpu, ref[0]))
        return res
    osel = oracle.block_select(q, k, t.s, t.block, t.alpha, rows=rows)
    nblk = osel.kept.shape[-1]
    gk = unpack_words(np.asarray(load("%s_%d_bits.npy" % (t.path, t.s))[:, hs]), nblk)[None]  # [1, R, G, nblk]
    diff = gk != osel.kept
    res["bad_pairs"] = int((diff & ~osel.near_pairs).sum())
    res["near_rows"] = int(osel.near.sum())
    res["rows_flipped"] = int(diff.any(axis=-1).sum())
    res["rows_total"] = int(osel.near.size)
    if res["bad_pairs"]:
        ref, _ = oracle.sparse(q, k, v, t.s, t.block, t.alpha, sel=osel)
    else:
        ref, _, _ = oracle.sparse_for_selection(q, k, v, t.s, t.block, t.alpha, gk, rows=rows)
    res.update(_err_stats(gpu, ref[0]))
    # the near rows' own errors (their outputs are held to the same bar)
    near = osel.near[0]
    if near.any():
        e = np.abs(gpu.astype(np.float64) - ref[0])[near]
        res["near_max"] = float(e.max())
    return res


def run_tasks(tasks, workers: int | None = None) -> list:
    """Runs the tasks in a spawned pool (heaviest first); returns their results."""
    workers = workers or os.cpu_count() or 1
    tasks = sorted(tasks, key=lambda t: -(t.s + t.C) * (1 if t.path == "sparse" else 4))
    saved = {k: os.environ.get(k) for k in _BLAS_ENV}
    for k in _BLAS_ENV:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(min(workers, len(tasks))) as pool:
            return pool.map(run_task, tasks, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def summarize(results) -> dict:
    """Per (path, chunk): max and mean |gpu - oracle| over the chunk's sampled rows and all heads."""
    out = {}
    for r in results:
        key = (r["path"], r["s"])
        a = out.setdefault(key, {"n": 0, "sum": 0.0, "max": 0.0, "finite": True, "bad_pairs": 0,
                                 "near_rows": 0, "rows_flipped": 0, "rows_total": 0, "near_max": 0.0})
        a["n"] += r["n"]
        a["sum"] += r["sum"]
        a["max"] = max(a["max"], r["max"])
        a["finite"] &= r["finite"]
        for f in ("bad_pairs", "near_rows", "rows_flipped", "rows_total"):
            a[f] += r.get(f, 0)
        a["near_max"] = max(a["near_max"], r.get("near_max", 0.0))
    for a in out.values():
        a["mean"] = a["sum"] / max(1, a["n"])
    return out
