"""The seeded input generator: determinism, statistics, subsets (CPU)."""

import math

import torch

from block_diffusion_lm_denoise_b300 import synth


def test_normal_is_deterministic_and_has_the_requested_moments():
    a = synth.normal((1 << 16,), 0.5, 7, "x", dtype=torch.float32)
    b = synth.normal((1 << 16,), 0.5, 7, "x", dtype=torch.float32)
    c = synth.normal((1 << 16,), 0.5, 8, "x", dtype=torch.float32)
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert abs(a.mean().item()) < 0.01
    assert abs(a.std().item() - 0.5) < 0.01
    assert a.abs().max().item() <= 0.5 * math.sqrt(12.0) + 1e-6   # Irwin-Hall bound


def test_bf16_output_is_the_rounded_float32_draw():
    a = synth.normal((4096,), 1.0, 3, "y", dtype=torch.float32)
    b = synth.normal((4096,), 1.0, 3, "y", dtype=torch.bfloat16)
    assert torch.equal(a.to(torch.bfloat16), b)


def test_kv_subset_equals_rows_of_the_full_tensor():
    full = synth.normal((5, 2, 7, 4), 1.0, 11, "kv")
    sub = synth.kv_subset((5, 2, 7, 4), [3, 0], 1.0, 11, "kv")
    assert torch.equal(sub[0], full[3]) and torch.equal(sub[1], full[0])


def test_uniform_integers_bernoulli_ranges():
    u = synth.uniform((10000,), 0.2, 2.0, 1, "u")
    assert u.min().item() >= 0.2 and u.max().item() < 2.0
    assert abs(u.mean().item() - 1.1) < 0.03
    i = synth.integers((10000,), 1000, 1, "i")
    assert i.min().item() >= 0 and i.max().item() < 1000
    m = synth.bernoulli((10000,), 0.5, 1, "m")
    assert 0.47 < m.float().mean().item() < 0.53
