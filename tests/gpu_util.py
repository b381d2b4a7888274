"""Helpers shared by the GPU parity tests (upload of generator bits, error stats)."""
import numpy as np
import torch

MAX_ABS = 5e-3     # attention output bar: max |gpu - oracle|
MEAN_ABS = 5e-4    # attention output bar: mean |gpu - oracle|


def dev(bits: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).cuda()


def errors(gpu: torch.Tensor, ref: np.ndarray):
    e = np.abs(gpu.detach().float().cpu().double().numpy() - ref)
    return float(e.max()), float(e.mean())


def assert_close(gpu, ref, what=""):
    mx, mean = errors(gpu, ref)
    assert np.isfinite(mx), (what, "non-finite output")
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (what, mx, mean)
    return mx, mean


def sample_rows(C: int, n: int, seed: int) -> np.ndarray:
    """Seeded row sample: n random rows plus the last 128 rows and every 128-row tile boundary."""
    g = np.random.default_rng(seed)
    rows = set(g.choice(C, size=min(n, C), replace=False).tolist())
    rows.update(range(max(0, C - 128), C))
    for t in range(0, C, 128):
        rows.update({t, min(C - 1, t + 127)})
    return np.array(sorted(rows))
