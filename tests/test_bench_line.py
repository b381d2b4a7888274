"""bench.py's oracle arm on CPU: one JSON line with the contract's keys, on the same metric and
workload as the GPU arm, reporting what it ran (cores, sample) and no host<->device traffic."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench
    args = type("A", (), {"warmup": 0, "steps": 1})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
                "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 1 and line["n_gpus"] == 1
    assert "32K" in line["config"]["workload"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert "query rows" in cb["sample"] and "cores" in cb["host"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_traffic_stamp_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    """The stored ncu traffic figure is voided by a change to the kernel's code, not by an
    edited comment or re-indented line."""
    import shutil
    import bench
    src = os.path.join(bench.ROOT, "long_context_prefill_chunked_gb300", "csrc")
    dst = tmp_path / "long_context_prefill_chunked_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in ("attn_fwd.cu", "kernels.cuh", "ptx.cuh"):
        shutil.copy(os.path.join(src, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    p = dst / "ptx.cuh"
    text = p.read_text()
    p.write_text("// an added comment\n/* and a block\n comment */\n" + text.replace("\n", "\n  ", 3))
    assert bench.kernel_source_hash() == h0
    p.write_text(text + "\nstatic int pf_probe_extra_symbol;\n")
    assert bench.kernel_source_hash() != h0
