"""Benchmark: long-context prefill attention at 32K tokens on GB300.

One step = one 32K-token prompt (32 query heads, 8 KV heads, head_dim 128,
bf16, planted block structure) through the whole path:
  * dense chunked prefill: 8 chunks of 4096 rows, each causal over the
    previous chunks' K/V, emitting the chunk's K/V into a head-major cache;
  * block-sparse prefill of the same prompt: block index (pool, score,
    select, compact) + exact kept blocks with the pooled correction.
The metric is dense-equivalent TFLOP/s: 4 * Hq * d * (causal query-key pairs of
the prompt), counted once per step although both paths compute it, over the
step time; each path's own TFLOP/s and tokens/s are reported beside it.  The same
run also measures the 128K-token prompt (32 chunks of 4096 over a growing
history) through both paths (``long_128k``) and times the oracle in full on
the three small workloads (``oracle_full``).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun) every rank runs an independent replica (weak scaling);
time is the max over ranks.  ``--impl reference`` times the float64 CPU oracle
instead (bounded sample per step).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attention TFLOP/s (dense-equiv) & tokens/s at 32K; % of bf16 TC peak"
N_TOK, HQ, HKV, D, CHUNK, BLOCK, ALPHA = 32768, 32, 8, 128, 4096, 128, 0.1
WORKLOAD = ("32K-token prompt, 32q/8kv heads, d128, bf16, planted blocks (beta %g); dense chunked "
            "prefill 8x4096 causal + block-sparse prefill (block 128, alpha 0.1)")


def pairs_causal(C, s):
    return C * s + C * (C + 1) // 2


def flops_equiv(C, s, Hq=HQ, d=D):
    return 4.0 * Hq * d * pairs_causal(C, s)


def kernel_source_hash():
    """sha256 over the code of the sources that define the dense attention kernel, comments and
    whitespace removed (a stored ncu traffic figure is only reported while the code it was
    measured on is unchanged; editing a comment does not change the kernel)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("attn_fwd.cu", "kernels.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "long_context_prefill_chunked_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)   # block comments
        src = re.sub(r"//[^\n]*", "", src)                 # line comments (no string here holds //)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()


def max_over_ranks(value_ms, device, world):
    """The slowest rank's time: every rank contributes its own, all receive the maximum."""
    if world <= 1:
        return value_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([value_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_rank, ms_per_step, world):
    """Whole-job throughput: every rank processed flops_per_rank in the slowest rank's time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return j, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.gpu = gpu_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------- oracle legs
def oracle_sample_rate(w, seconds, seed=0):
    """Time the float64 oracle on sampled rows of the last 4096-row chunk, each row through both
    paths (dense over its 28672-token history + chunk, and block-sparse); a row's dense-equivalent
    work is counted once.  Returns (TFLOP/s equiv, detail)."""
    import oracle
    g = np.random.default_rng(seed)
    s_last = N_TOK - CHUNK
    q_last = w.f64(w.q[:, s_last:])
    kh, vh = w.f64(w.k[:, :s_last]), w.f64(w.v[:, :s_last])
    kc, vc = w.f64(w.k[:, s_last:]), w.f64(w.v[:, s_last:])
    k_all, v_all = w.f64(w.k), w.f64(w.v)
    flops = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        rows = np.sort(g.choice(CHUNK, size=16, replace=False))
        oracle.dense(q_last, kh, vh, kc, vc, s_last, rows=rows)
        oracle.sparse(q_last, k_all, v_all, s_last, BLOCK, ALPHA, rows=rows)
        flops += sum(4.0 * HQ * D * (s_last + r + 1) for r in rows)
        rows_done += 16
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, {"rows": rows_done, "seconds": dt, "threads": _blas_threads()}


def oracle_full_timings():
    """The oracle timed in full on the three small workloads (every row, every head), and the
    per-(row, head, key) cost of the largest one extrapolated to the 32K and 128K prompts."""
    import oracle
    import prefill_inputs as pi
    res = {}
    w1 = pi.config(1)
    t0 = time.perf_counter()
    oracle.dense(*(w1.f64(x) for x in w1.chunk_views(0)), 0, mask=pi.causal_mask(256, 0, np.float64))
    res["config1_s"] = time.perf_counter() - t0
    w2 = pi.config(2)
    t0 = time.perf_counter()
    pairs2 = 0
    for s in w2.starts:
        oracle.dense(*(w2.f64(x) for x in w2.chunk_views(s)), s, mask=pi.causal_mask(w2.chunk, s, np.float64))
        pairs2 += w2.chunk * (s + w2.chunk)
    res["config2_s"] = time.perf_counter() - t0
    w3 = pi.config(3)
    mask, _ = pi.indexer_fold_mask(w3.seed, w3.chunk, 8192)
    t0 = time.perf_counter()
    oracle.dense(*(w3.f64(x) for x in w3.chunk_views(8192)), 8192, mask=mask.astype(np.float64))
    res["config3_s"] = time.perf_counter() - t0
    per_elem = res["config2_s"] / (pairs2 * w2.Hq)           # seconds per (row, head, key)
    causal = lambda n, c: sum(c * s + c * (c + 1) // 2 for s in range(0, n, c))
    res["extrapolated_32k_dense_s"] = per_elem * HQ * causal(N_TOK, CHUNK)
    res["extrapolated_128k_dense_s"] = per_elem * HQ * causal(131072, CHUNK)
    res["note"] = ("configs 1-3 timed in full (every row and head, explicit masks); the 32K and 128K "
                   "figures are EXTRAPOLATED from config 2's cost per (row, head, key), not run")
    res["cores"] = _blas_threads()
    return res


def _blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max((i.get("num_threads", 1) for i in info), default=os.cpu_count())
    except Exception:
        return os.cpu_count()


def host_cpu():
    """The host CPU as /proc/cpuinfo names it (x86 'model name', Arm implementer and part),
    with the architecture; the oracle's timing is only meaningful beside it."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ":" in ln:
                    k, v = ln.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        model = fields["model name"]
    elif "CPU part" in fields:
        model = "implementer %s part %s" % (fields.get("CPU implementer", "?"), fields["CPU part"])
    else:
        model = platform.processor() or "unknown"
    return "%s (%s, %d logical cores)" % (model, platform.machine(), os.cpu_count() or 0)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import prefill_inputs as pi
    w = pi.config(4)
    per_step = []
    for i in range(args.warmup + args.steps):
        v, det = oracle_sample_rate(w, 2.0, seed=i)
        if i >= args.warmup:
            per_step.append((v, det))
    value = statistics.mean(v for v, _ in per_step)
    rows = sum(d["rows"] for _, d in per_step)
    secs = sum(d["seconds"] for _, d in per_step)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": WORKLOAD % pi.PLANT_BETA},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": per_step[0][1]["threads"],
                         "kind": "oracle", "host": host_cpu(),
                         "sample": "%d query rows x 32 heads of the last 4096-row chunk, each through "
                                   "the dense and the block-sparse oracle (work counted once), float64 "
                                   "numpy oracle" % rows},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- profiling cases
def run_case(args):
    """Small cases for ncu: the last dense chunk of the 32K prompt (K/V 134 MB, larger than L2)
    or the 32K block-sparse pair.  Prints per-iteration times; not a bench line."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import long_context_prefill_chunked_gb300 as pfx
    import prefill_inputs as pi
    to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    if args.case == "mask-config2":
        # config 2: three 4096-row chunks (16q/8kv, d128) at starts 0 / 4096 / 8192, each under an
        # explicit fp32 0 / -30000 causal mask, K/V re-emitted into a head-major cache
        w2 = pi.config(2)
        Q, K, V = (to_dev(x) for x in (w2.q, w2.k, w2.v))
        V16 = torch.empty(V.shape, dtype=torch.float16, device="cuda")  # v kept in fp16, chunk by chunk
        masks = [torch.from_numpy(pi.causal_mask(w2.chunk, s)).cuda() for s in w2.starts]
        ck = torch.empty((1, w2.Hkv, w2.N, w2.d), dtype=torch.bfloat16, device="cuda")
        cv = torch.empty((1, w2.Hkv, w2.N, w2.d), dtype=torch.float16, device="cuda")

        def run():
            for s, m in zip(w2.starts, masks):
                c = w2.chunk
                pfx.to_f16(V[:, s:s + c], out=V16[:, s:s + c])
                pfx.attn_dense(Q[:, s:s + c], K[:, :s], V16[:, :s], K[:, s:s + c], V16[:, s:s + c], s, mask=m,
                               out_k=ck[:, :, s:s + c], out_v=cv[:, :, s:s + c])
        flops = sum(4.0 * w2.Hq * w2.d * (w2.chunk * s + w2.chunk * (w2.chunk + 1) // 2) for s in w2.starts)
        return _time_case(args, pfx, run, flops, 0)
    if args.case in ("indexed-config3", "mask-config3"):
        # a 4096-row chunk over an 8192-token history (16q/8kv, d128), 512 compressed blocks of
        # 4 keys kept per query: as keep lists, or folded into an fp32 0 / -30000 mask
        w3 = pi.config(3)
        s = 8192
        q, kh, vh, kc, vc = (to_dev(x) for x in w3.chunk_views(s))
        vh16 = pfx.to_f16(vh.contiguous())  # the history's v, converted by the earlier chunks
        vc16 = torch.empty(vc.shape, dtype=torch.float16, device="cuda")
        vc = vc.contiguous()
        mask, kept = pi.indexer_fold_mask(w3.seed, w3.chunk, s)
        if args.case == "indexed-config3":
            idx = torch.from_numpy(np.stack(kept).astype(np.int32)).cuda()
            cnt = torch.full((w3.chunk,), idx.shape[1], dtype=torch.int32, device="cuda")

            def run():
                pfx.to_f16(vc, out=vc16)
                pfx.attn_indexed(q, kh, vh16, kc, vc16, s, idx, cnt, 4)
        else:
            m = torch.from_numpy(mask).cuda()

            def run():
                pfx.to_f16(vc, out=vc16)
                pfx.attn_dense(q, kh, vh16, kc, vc16, s, mask=m)
        return _time_case(args, pfx, run, 4.0 * w3.Hq * w3.d * (w3.chunk * s + w3.chunk * (w3.chunk + 1) // 2), s)
    w = pi.config(5 if args.case == "sparse-128k-chunk" else 4)
    if args.case == "sparse-128k-chunk":
        # the last 4096-row chunk of the 128K planted prompt: selection and block-sparse
        # attention against a 131072-key history (K/V 268 MB each, beyond L2)
        s = w.N - CHUNK
        K, V, Q = to_dev(w.k), to_dev(w.v), to_dev(w.q[:, s:])
        V16 = pfx.to_f16(V)  # the history's v, converted by the earlier chunks
        sel = pfx.alloc_selection(Q, K, s)
        pooled = pfx.alloc_pooled(Q, K, s)
        out = torch.empty((1, CHUNK, HQ, D), dtype=torch.float32, device="cuda")

        def run():
            pfx.block_index(Q, K, s, BLOCK, ALPHA, sel=sel)
            pfx.to_f16(V[:, s:], out=V16[:, s:])
            pfx.attn_sparse(Q, K, V16, s, sel, pooled=pooled, out=out)
        return _time_case(args, pfx, run, flops_equiv(CHUNK, s), s)
    s = args.start
    if s % CHUNK != 0 or not 0 <= s < N_TOK:
        raise SystemExit("--start must be a multiple of %d below %d" % (CHUNK, N_TOK))
    K, V = to_dev(w.k), to_dev(w.v)
    V16 = pfx.to_f16(V)  # v kept in fp16 as in the bench step (the history converted by earlier chunks)
    Q = to_dev(w.q[:, s:s + CHUNK]) if args.case == "dense-chunk" else to_dev(w.q)
    if args.case == "dense-chunk":
        # as in the bench step: the chunk's v converted, its K/V re-emitted into a head-major cache
        out = torch.empty((1, CHUNK, HQ, D), dtype=torch.float32, device="cuda")
        ck = torch.empty((1, HKV, CHUNK, D), dtype=torch.bfloat16, device="cuda")
        cv = torch.empty((1, HKV, CHUNK, D), dtype=torch.float16, device="cuda")

        def run():
            pfx.to_f16(V[:, s:s + CHUNK], out=V16[:, s:s + CHUNK])
            pfx.attn_dense(Q, K[:, :s], V16[:, :s], K[:, s:s + CHUNK], V16[:, s:s + CHUNK], s, out=out,
                           out_k=ck, out_v=cv)
        flops = flops_equiv(CHUNK, s)
    else:
        sel = pfx.alloc_selection(Q, K, 0)
        pooled = pfx.alloc_pooled(Q, K, 0)
        out = torch.empty((1, N_TOK, HQ, D), dtype=torch.float32, device="cuda")
        # sparse-shared: the Metal port's KV-group shared selection (share_group_kernel)
        rules = pfx.KeepRules(share_kv_group=1) if args.case == "sparse-shared" else None

        def run():
            pfx.block_index(Q, K, 0, BLOCK, ALPHA, sel=sel, rules=rules)
            pfx.to_f16(V, out=V16)
            pfx.attn_sparse(Q, K, V16, 0, sel, pooled=pooled, out=out)
        flops = flops_equiv(N_TOK, 0)
    return _time_case(args, pfx, run, flops, s if args.case == "dense-chunk" else 0)


def _time_case(args, pfx, run, flops, start):
    import torch
    for _ in range(args.warmup):
        run()
    pfx.stream_status()
    times = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    pfx.stream_status()
    print(json.dumps({"case": args.case, "start": start, "ms": times,
                      "tflops_equiv": flops / (min(times) * 1e-3) / 1e12}))
    return 0


# ---------------------------------------------------------------------------- 128K record
def run_long_128k(pfx, dev, reps=3, warmup=1):
    """The 128K-token planted prompt (32q/8kv, d128, bf16) as a chunked prefill: 32 chunks of 4096
    rows over a growing history (0 .. 126,976 rows), each chunk through dense causal prefill
    (emitting its K/V into a head-major cache, tail-split workspace on) and, separately, through
    block-sparse prefill (block index + sparse attention with the pooled correction, block 128,
    alpha 0.1; one pooled-key buffer and workspace for the prompt, each chunk pooling only its
    own blocks).  CUDA events per call on the launching stream; the median over `reps` passes
    (inputs are 1.5 GB, far beyond L2).  The block-sparse prefill is also timed pipelined: each
    chunk's block index on a low-priority stream ahead of the sparse attention on a high-priority
    one (wall time, `sparse_pipelined_ms`).  Skip share is weighted by dense work: per (head, query
    tile) the dense path runs its off-diagonal key tiles plus half a diagonal tile, the sparse
    path its kept off-diagonal tiles plus the same half (pooled tiles not counted)."""
    import torch
    import prefill_inputs as pi
    w = pi.config(5)
    N, C = w.N, w.chunk
    to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)
    Q, K, V = to_dev(w.q), to_dev(w.k), to_dev(w.v)
    starts = w.starts
    out = torch.empty((1, C, HQ, D), dtype=torch.float32, device=dev)
    cache_k = torch.empty((1, HKV, N, D), dtype=torch.bfloat16, device=dev)
    cache_v = torch.empty((1, HKV, N, D), dtype=torch.float16, device=dev)
    v16_d = torch.empty(V.shape, dtype=torch.float16, device=dev)  # each path's fp16 v, chunk by chunk
    v16_s = torch.empty_like(v16_d)
    # one pooled-key buffer and one sparse workspace for the whole prompt: each chunk pools only
    # its own blocks (the history's block means do not change)
    kbar = pfx.alloc_kbar(Q[:, :C], K, N, BLOCK)
    pooled = pfx.alloc_pooled(Q[:, :C], K, 0, BLOCK, max_keys=N)
    sels = [pfx.alloc_selection(Q[:, s:s + C], K[:, :s + C], s, BLOCK, kbar=kbar, pooled_blocks=s // BLOCK)
            for s in starts]
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    dense_t, index_t, attn_t = [], [], []
    for it in range(warmup + reps):
        e = {"d": [(ev(), ev()) for _ in starts], "i": [(ev(), ev()) for _ in starts],
             "a": [(ev(), ev()) for _ in starts]}
        for i, s in enumerate(starts):
            e["d"][i][0].record(stream)
            pfx.to_f16(V[:, s:s + C], out=v16_d[:, s:s + C], stream=stream)
            pfx.attn_dense(Q[:, s:s + C], K[:, :s], v16_d[:, :s], K[:, s:s + C], v16_d[:, s:s + C], s, out=out,
                           out_k=cache_k[:, :, s:s + C], out_v=cache_v[:, :, s:s + C], stream=stream)
            e["d"][i][1].record(stream)
        for i, s in enumerate(starts):
            q = Q[:, s:s + C]
            e["i"][i][0].record(stream)
            pfx.block_index(q, K[:, :s + C], s, BLOCK, ALPHA, sel=sels[i], stream=stream)
            e["i"][i][1].record(stream)
            e["a"][i][0].record(stream)
            pfx.to_f16(V[:, s:s + C], out=v16_s[:, s:s + C], stream=stream)
            pfx.attn_sparse(q, K[:, :s + C], v16_s[:, :s + C], s, sels[i], block=BLOCK, pooled=pooled, out=out,
                            stream=stream)
            e["a"][i][1].record(stream)
        torch.cuda.synchronize(dev)
        if it >= warmup:
            dense_t.append([a.elapsed_time(b) for a, b in e["d"]])
            index_t.append([a.elapsed_time(b) for a, b in e["i"]])
            attn_t.append([a.elapsed_time(b) for a, b in e["a"]])
    pfx.stream_status(stream)
    # the same block-sparse prefill pipelined as a caller would run it: the block index of each
    # chunk on a low-priority stream, the v conversion and sparse attention on a high-priority one
    # (attention i waits for index i only), so the next chunks' index kernels take the SMs the
    # attention kernel leaves idle in its last wave.  Wall time from the first call to the last.
    hi = torch.cuda.Stream(dev, priority=-1)
    lo = torch.cuda.Stream(dev, priority=0)
    pipe_t = []
    for it in range(warmup + reps):
        e0, e1 = ev(), ev()
        done = [torch.cuda.Event() for _ in starts]
        e0.record(hi)
        lo.wait_event(e0)
        for i, s in enumerate(starts):
            q = Q[:, s:s + C]
            pfx.block_index(q, K[:, :s + C], s, BLOCK, ALPHA, sel=sels[i], stream=lo)
            done[i].record(lo)
            pfx.to_f16(V[:, s:s + C], out=v16_s[:, s:s + C], stream=hi)
            hi.wait_event(done[i])
            pfx.attn_sparse(q, K[:, :s + C], v16_s[:, :s + C], s, sels[i], block=BLOCK, pooled=pooled, out=out,
                            stream=hi)
        e1.record(hi)
        torch.cuda.synchronize(dev)
        if it >= warmup:
            pipe_t.append(e0.elapsed_time(e1))
    pfx.stream_status(hi)
    pfx.stream_status(lo)
    t_pipe = statistics.median(pipe_t)
    med = lambda runs: statistics.median(sum(r) for r in runs)
    t_dense, t_index, t_attn = med(dense_t), med(index_t), med(attn_t)
    t_sparse = t_index + t_attn
    dense_w = sparse_w = 0.0
    for s, sel in zip(starts, sels):
        tc = sel.tile_cnt.cpu().numpy().astype(np.float64)             # [1, Hq, nqt]
        ob = s // BLOCK + np.arange(tc.shape[-1])
        dense_w += HQ * (ob + 0.5).sum()
        sparse_w += (tc - 1 + 0.5).sum()
    skip = 1.0 - sparse_w / dense_w
    flops = sum(flops_equiv(C, s) for s in starts)
    del Q, K, V, cache_k, cache_v, sels, kbar, pooled, out
    torch.cuda.empty_cache()
    return {
        "workload": "128K-token prompt, 32q/8kv, d128, bf16, planted blocks (beta %g), 32 chunks x 4096 "
                    "over a growing history; block 128, alpha 0.1" % w.beta,
        "dense_ms": t_dense, "dense_tflops": flops / (t_dense * 1e-3) / 1e12,
        "dense_tokens_per_s": N / (t_dense * 1e-3),
        "sparse_ms": t_sparse, "sparse_index_ms": t_index, "sparse_attn_ms": t_attn,
        "sparse_tflops_equiv": flops / (t_sparse * 1e-3) / 1e12, "sparse_tokens_per_s": N / (t_sparse * 1e-3),
        "skip_share_flop_weighted": skip,
        "speedup": t_dense / t_sparse,
        "efficiency": (t_dense / t_sparse) * (1.0 - skip),
        "efficiency_note": "(t_dense / t_sparse) * (1 - skip); 1 = sparse time exactly in proportion to "
                           "the dense work it keeps",
        "sparse_pipelined_ms": t_pipe,
        "sparse_pipelined_tflops_equiv": flops / (t_pipe * 1e-3) / 1e12,
        "efficiency_pipelined": (t_dense / t_pipe) * (1.0 - skip),
        "pipelined_note": "wall time of the block-sparse prefill with each chunk's block index on a "
                          "low-priority stream and its attention on a high-priority one (attention i "
                          "waits for index i); sparse_ms is the sum of the per-call times on one stream",
        "dense_ms_per_chunk": [statistics.median(r[i] for r in dense_t) for i in range(len(starts))],
        "sparse_ms_per_chunk": [statistics.median(a[i] + b[i] for a, b in zip(index_t, attn_t))
                                for i in range(len(starts))],
        "sparse_index_ms_per_chunk": [statistics.median(r[i] for r in index_t) for i in range(len(starts))],
        "reps": reps,
    }


TRAFFIC_CMD = ("python bench.py --steps 1 --warmup 3 --no-cpu-baseline --no-long --e2e-steps 1 && "
               "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
               "--clock-control none --print-units base --kernel-name-base demangled "
               "-k 'regex:attn_fwd_kernel<\\(int\\)0' -s 0 -c 8 --csv --log-file traffic.csv "
               "python bench.py --steps 1 --warmup 3 --no-cpu-baseline --no-long --e2e-steps 1 && "
               "python bench.py --write-traffic traffic.csv")


def write_traffic(csv_path):
    """Turn the ncu capture of TRAFFIC_CMD (the eight dense causal launches of the first warm-up
    step, one per 4096-row chunk in order) into profiles/attn_dense_traffic.json, stamped with the
    kernel sources' hash so that the bench reports it only while the kernel is unchanged."""
    import csv
    import re
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9,
             "ns": 1e-6, "nsecond": 1e-6, "us": 1e-3, "usecond": 1e-3, "ms": 1.0, "msecond": 1.0, "s": 1e3,
             "second": 1e3}
    launches = {}
    with open(csv_path) as fh:
        rows = [ln for ln in fh if ln.startswith('"')]
    for r in csv.DictReader(rows):
        if not re.search(r"attn_fwd_kernel<(\(int\))?0[,>]", r["Kernel Name"]):  # mode 0: causal
            continue
        v = float(r["Metric Value"].replace(",", "")) * scale[r["Metric Unit"]]
        launches.setdefault(int(r["ID"]), {})[r["Metric Name"]] = v
    ids = sorted(launches)
    if len(ids) != len(range(0, N_TOK, CHUNK)):
        raise SystemExit("expected %d dense launches in %s, found %d" % (N_TOK // CHUNK, csv_path, len(ids)))
    per = []
    for i, start in zip(ids, range(0, N_TOK, CHUNK)):
        m = launches[i]
        # algorithmic: Q, the chunk's K / V and the history's K / V read once (bf16), fp32 O written
        alg = 2 * CHUNK * HQ * D + 2 * 2 * (start + CHUNK) * HKV * D + 4 * CHUNK * HQ * D
        per.append({"start": start, "dram_read": int(m["dram__bytes_read.sum"]),
                    "dram_write": int(m["dram__bytes_write.sum"]), "algorithmic": alg,
                    "ncu_ms": round(m["gpu__time_duration.sum"], 6)})
    rec = {
        "kernel": "attn_fwd_kernel<0> (dense causal)",
        "workload": "32K prompt, 8 chunks of 4096 rows, 32q/8kv, d128, bf16 in, fp32 out",
        "bytes_per_launch": int(round(sum(x["dram_read"] + x["dram_write"] for x in per) / len(per))),
        "source_sha256": kernel_source_hash(),
        "note": "dram__bytes_read.sum + dram__bytes_write.sum of the 8 causal launches of one step (the "
                "first warm-up step of the command below), averaged; writes undercount the fp32 output "
                "because dirty lines can still sit in L2 when the kernel ends",
        "command": TRAFFIC_CMD,
        "per_launch": per,
    }
    with open(os.path.join(ROOT, "profiles", "attn_dense_traffic.json"), "w") as fh:
        json.dump(rec, fh, indent=1)
        fh.write("\n")
    print(json.dumps({"bytes_per_launch": rec["bytes_per_launch"], "launches": len(per)}))


# ---------------------------------------------------------------------------- ours
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30,
                    help="steps in the end-to-end window (one pipeline fill and one drain amortised over them)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the 128K-token record")
    ap.add_argument("--long-reps", type=int, default=3)
    ap.add_argument("--case", default="full", choices=["full", "dense-chunk", "sparse", "sparse-shared",
                                                       "sparse-128k-chunk", "indexed-config3", "mask-config3",
                                                       "mask-config2"],
                    help="profiling cases, timings only: dense-chunk (one 4096-row chunk at "
                         "--start, K/V re-emitted into a cache), sparse (the 32K block-sparse pair), "
                         "sparse-shared (the same with KV-group shared selection), sparse-128k-chunk "
                         "(the pair for the last 4096-row chunk of the 128K prompt), indexed-config3 / "
                         "mask-config3 (config 3's selection as keep lists / as a folded mask), "
                         "mask-config2 (config 2's three chunks under explicit causal masks)")
    ap.add_argument("--start", type=int, default=N_TOK - CHUNK,
                    help="dense-chunk case: the chunk's first token (a multiple of 4096)")
    ap.add_argument("--write-traffic", metavar="CSV",
                    help="write profiles/attn_dense_traffic.json from an ncu capture (no GPU work)")
    args = ap.parse_args()
    if args.write_traffic:
        return write_traffic(args.write_traffic)
    if args.impl == "reference":
        return run_reference(args)
    if args.case != "full":
        return run_case(args)

    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    import long_context_prefill_chunked_gb300 as pfx
    import prefill_inputs as pi

    w = pi.config(4)
    to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)
    Q, K, V = to_dev(w.q), to_dev(w.k), to_dev(w.v)
    out_d = torch.empty((1, N_TOK, HQ, D), dtype=torch.float32, device=dev)
    out_s = torch.empty_like(out_d)
    cache_k = torch.empty((1, HKV, N_TOK, D), dtype=torch.bfloat16, device=dev)
    cache_v = torch.empty((1, HKV, N_TOK, D), dtype=torch.float16, device=dev)  # v cached in fp16
    sel = pfx.alloc_selection(Q, K, 0, BLOCK)
    pooled = pfx.alloc_pooled(Q, K, 0, BLOCK)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    starts = list(range(0, N_TOK, CHUNK))

    def mk():
        return torch.cuda.Event(enable_timing=True)

    # v is kept in fp16 (the v_f16 mode): each path converts the bf16 v it reads once
    # (pf_convert_f16, inside the step) instead of every CTA converting every v tile it loads
    v16_d = torch.empty(V.shape, dtype=torch.float16, device=dev)  # the dense path's fp16 v
    v16_s = torch.empty_like(v16_d)                                  # the block-sparse path's

    def step(q, k, v, ev=None, outs=None):
        o_d, o_s, c_k, c_v = outs if outs is not None else (out_d, out_s, cache_k, cache_v)
        for i, s in enumerate(starts):
            if ev is not None:
                ev["dense"][i][0].record(stream)
            pfx.to_f16(v[:, s:s + CHUNK], out=v16_d[:, s:s + CHUNK], stream=stream)
            pfx.attn_dense(q[:, s:s + CHUNK], k[:, :s], v16_d[:, :s], k[:, s:s + CHUNK], v16_d[:, s:s + CHUNK],
                           s, out=o_d[:, s:s + CHUNK], out_k=c_k[:, :, s:s + CHUNK],
                           out_v=c_v[:, :, s:s + CHUNK], stream=stream)
            if ev is not None:
                ev["dense"][i][1].record(stream)
        if ev is not None:
            ev["index"][0].record(stream)
        pfx.block_index(q, k, 0, BLOCK, ALPHA, sel=sel, stream=stream)
        if ev is not None:
            ev["index"][1].record(stream)
            ev["sparse"][0].record(stream)
        pfx.to_f16(v, out=v16_s, stream=stream)
        pfx.attn_sparse(q, k, v16_s, 0, sel, block=BLOCK, pooled=pooled, out=o_s, stream=stream)
        if ev is not None:
            ev["sparse"][1].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step(Q, K, V)
    pfx.stream_status(stream)

    evs = [{"dense": [(mk(), mk()) for _ in starts], "index": (mk(), mk()), "sparse": (mk(), mk()),
            "step": (mk(), mk())} for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    pfx.launch_count(reset=True)
    for i in range(args.steps):
        flush.zero_()                       # L2 flush between steps (outside the step window)
        evs[i]["step"][0].record(stream)
        step(Q, K, V, evs[i])
        evs[i]["step"][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = pfx.launch_count()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    pfx.stream_status(stream)

    step_ms = [e["step"][0].elapsed_time(e["step"][1]) for e in evs]
    dense_ms = [[a.elapsed_time(b) for a, b in e["dense"]] for e in evs]
    index_ms = [e["index"][0].elapsed_time(e["index"][1]) for e in evs]
    sparse_ms = [e["sparse"][0].elapsed_time(e["sparse"][1]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms), dev, world)
    ms_step = total_ms / args.steps

    f_dense = sum(flops_equiv(CHUNK, s) for s in starts)
    f_sparse = flops_equiv(N_TOK, 0)
    # the step computes the prompt's causal attention twice (dense, then block-sparse): its
    # dense-equivalent work and its tokens are counted once
    f_prompt = f_dense
    value = weak_scaling_value(f_prompt, ms_step, world)
    tokens_per_s = world * N_TOK / (ms_step * 1e-3)

    # dominant kernel: the dense attention launches (8 per step)
    d_ms = sum(map(sum, dense_ms)) / args.steps
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = f_dense / (d_ms * 1e-3) / 1e12
    traffic, traffic_note = None, "no ncu capture on file"
    tpath = os.path.join(ROOT, "profiles", "attn_dense_traffic.json")
    if os.path.exists(tpath):
        tj = json.load(open(tpath))
        if tj.get("source_sha256") == kernel_source_hash():
            traffic, traffic_note = tj.get("bytes_per_launch"), tj.get("note")
        else:
            traffic_note = "kernel source changed since the ncu capture"

    tc = sel.tile_cnt.cpu().numpy().astype(np.float64)
    n_qt = tc.shape[-1]
    cand = HQ * sum(range(n_qt))
    skip_tiles = 1.0 - (tc - 1).sum() / cand

    # e2e: host buffers in, host buffers out, through the same public API.  Pipelined as a
    # serving loop would run it: two buffer sets, the next step's H2D and the previous step's
    # D2H on their own streams while this step computes; the window runs from the first H2D
    # to the last D2H.
    hq = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).pin_memory()
    hk = torch.from_numpy(w.k.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(w.v.view(np.int16)).view(torch.bfloat16).pin_memory()
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    sets = []
    for b in range(2):
        dins = (torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V))
        douts = (out_d, out_s, cache_k, cache_v) if b == 0 else tuple(torch.empty_like(t) for t in
                                                                         (out_d, out_s, cache_k, cache_v))
        houts = tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in douts)
        sets.append({"in": dins, "out": douts, "host": houts, "in_ready": torch.cuda.Event(),
                     "comp_done": torch.cuda.Event(), "out_done": torch.cuda.Event(), "used": False})

    def e2e_step(i):
        bs = sets[i % 2]
        with torch.cuda.stream(h2d_stream):
            if bs["used"]:
                h2d_stream.wait_event(bs["comp_done"])      # step i-2 has read these inputs
            for d, h in zip(bs["in"], (hq, hk, hv)):
                d.copy_(h, non_blocking=True)
            bs["in_ready"].record(h2d_stream)
        stream.wait_event(bs["in_ready"])
        if bs["used"]:
            stream.wait_event(bs["out_done"])             # step i-2's outputs are on the host
        step(*bs["in"], outs=bs["out"])
        bs["comp_done"].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(bs["comp_done"])
            for hbuf, d in zip(bs["host"], bs["out"]):
                hbuf.copy_(d, non_blocking=True)
            bs["out_done"].record(d2h_stream)
        bs["used"] = True

    for i in range(2):                      # untimed warm-up of both buffer sets
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = mk(), mk()
    e0.record(stream)
    h2d_stream.wait_event(e0)
    for i in range(args.e2e_steps):
        e2e_step(i)
    for bs in sets:
        stream.wait_event(bs["out_done"])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dev, world)
    pfx.stream_status(stream)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = sum(x.numel() * x.element_size() for x in sets[0]["host"])

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) Q/K/V with planted key blocks (no dataset)",
        "config": {"workload": WORKLOAD % w.beta, "tokens": N_TOK, "Hq": HQ, "Hkv": HKV, "head_dim": D,
                   "chunk": CHUNK, "block": BLOCK, "alpha": ALPHA, "out_dtype": "f32",
                   "v": "bf16 input; each path converts it to fp16 once inside the step (pf_convert_f16) "
                        "and its kernels read the fp16 v (P*V runs in fp16); the chunk cache keeps k bf16, v fp16",
                   "l2": "flushed between steps (256 MB write outside the step window)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tokens_per_s": tokens_per_s,
        "step_note": "one step = the 32K prompt through dense chunked prefill (8 x 4096) and through "
                     "block-sparse prefill; value and tokens_per_s count the prompt once per step; "
                     "each path's own rate is below",
        "dense_chunked_tflops": f_dense / (d_ms * 1e-3) / 1e12,
        "dense_chunked_tokens_per_s": N_TOK / (d_ms * 1e-3),
        "block_sparse_tflops_equiv": f_sparse / ((statistics.mean(index_ms) + statistics.mean(sparse_ms)) * 1e-3) / 1e12,
        "block_sparse_tokens_per_s": N_TOK / ((statistics.mean(index_ms) + statistics.mean(sparse_ms)) * 1e-3),
        "paths": {
            "dense_chunked": {"ms": sum(map(sum, dense_ms)) / args.steps,
                              "tflops_equiv": f_dense / (d_ms * 1e-3) / 1e12,
                              "tokens_per_s": N_TOK / (d_ms * 1e-3),
                              "ms_per_chunk": [statistics.mean(x[i] for x in dense_ms) for i in range(len(starts))]},
            "block_sparse": {"ms": statistics.mean(index_ms) + statistics.mean(sparse_ms),
                             "index_ms": statistics.mean(index_ms), "attn_ms": statistics.mean(sparse_ms),
                             "tflops_equiv": f_sparse / ((statistics.mean(index_ms) + statistics.mean(sparse_ms)) * 1e-3) / 1e12,
                             "skip_share_tiles": skip_tiles},
        },
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic, "traffic_note": traffic_note,
                     "kernel": "attn_fwd_kernel<causal> (8 launches per step; window includes the "
                               "chunk's two cache-layout copies)",
                     "peak_source": "%s bf16_tflops (burst)" % peak_src},
        "e2e": {"value": weak_scaling_value(f_prompt, e2e_ms, world), "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelining": "two buffer sets; step i+1's H2D and step i-1's D2H overlap step i on "
                              "their own streams; window from the first H2D to the last D2H"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if world == 1 and not args.no_long:
        line["long_128k"] = run_long_128k(pfx, dev, reps=args.long_reps)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, det = oracle_sample_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": det["threads"], "kind": "oracle",
                                "host": host_cpu(),
                                "sample": "%d query rows x 32 heads of the last 4096-row chunk (keys "
                                          "28672..32767) in %.1f s, each row through the dense and the "
                                          "block-sparse oracle (work counted once); float64 numpy oracle"
                                          % (det["rows"], det["seconds"])}
        line["oracle_full"] = oracle_full_timings()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
