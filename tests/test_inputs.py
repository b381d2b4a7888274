"""The seeded generators: rounding, reproducibility, the planted structure."""
import math

import numpy as np
import torch

import prefill_inputs as pi


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    x = (g.standard_normal(100000) * np.exp(g.uniform(-20, 20, 100000))).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]  # ties to even both ways
    ours = pi.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = pi.bits_to_f64(ours, "bf16")
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_f16_roundtrip_exact():
    g = np.random.default_rng(1)
    x = g.standard_normal(1000).astype(np.float32)
    bits = pi.f32_to_f16_bits(x)
    assert np.array_equal(pi.bits_to_f64(bits, "f16"), x.astype(np.float16).astype(np.float64))


def test_streams_reproducible_and_independent():
    a = pi.normal_f32(5, "q", (4, 8))
    b = pi.normal_f32(5, "q", (4, 8))
    c = pi.normal_f32(5, "k", (4, 8))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_causal_mask_shape_and_values():
    m = pi.causal_mask(3, 2)
    assert m.shape == (3, 5)
    assert m.tolist() == [[0, 0, 0, -30000, -30000], [0, 0, 0, 0, -30000], [0, 0, 0, 0, 0]]


def test_planted_structure_lifts_pooled_scores():
    w = pi.planted_workload("t", 3, 1, 4, 2, 64, 1024, 1024, "bf16", block=128, beta=8.0)
    assert w.q.shape == (1, 1024, 4, 64) and w.k.shape == (1, 1024, 2, 64)
    q, k = w.f64(w.q), w.f64(w.k)
    # the mean key of a planted block carries ~gamma along some query block's direction
    kb = k[0].reshape(8, 128, 2, 64).mean(axis=1)                  # [blocks, Hkv, d]
    qb = q[0].reshape(8, 128, 4, 64).mean(axis=1)                  # [blocks, Hq, d]
    s = np.einsum("qhd,khd->hqk", qb[:, ::2], kb) / math.sqrt(64)  # head 0 and 2 of each group
    # query block 7 has 4 planted blocks among 0..5: they stand ~beta*gamma/sqrt(d) = 4 above the rest
    top = np.sort(s[:, 7, :6], axis=1)
    assert (top[:, 2:].min(axis=1) - top[:, :2].max(axis=1)).min() > 1.0
