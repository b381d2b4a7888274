"""bench.py's multi-rank path on CPU: world_size 2 over gloo.  Every rank must end with the
slowest rank's time, the whole-job value must count every rank's work, and the oracle arm
must run on rank 0 only."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [3.0, 7.5][rank]                       # this rank's step time, ms
        slowest = bench.max_over_ranks(mine, torch.device("cpu"), world)
        value = bench.weak_scaling_value(8.8e12, slowest, world)
        # the reference arm: rank 0 prints one line, the others exit 0 without work
        buf = io.StringIO()
        args = type("A", (), {"warmup": 0, "steps": 1})()
        if rank != 0:
            with redirect_stdout(buf):
                rc = bench.run_reference(args)
        else:
            rc = 0
        dist.barrier()
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
            json.dump({"slowest": slowest, "value": value, "rc": rc, "printed": buf.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    for r in res:
        assert r["slowest"] == 7.5
        assert abs(r["value"] - 2 * 8.8e12 / 7.5e-3 / 1e12) < 1e-9
    assert res[1]["rc"] == 0 and res[1]["printed"] == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, None, 1) == 4.25
    assert bench.weak_scaling_value(1e12, 1000.0, 1) == 1.0     # 1 TFLOP in 1 s
