"""The seeded input generator: determinism and the recipe's statistics (CPU)."""
import numpy as np
import torch

import synth


def test_deterministic_and_counter_based():
    a = synth.weight(64, 96, seed=1, sigma=0.02, p=0.001, mult=20.0)
    b = synth.weight(64, 96, seed=1, sigma=0.02, p=0.001, mult=20.0)
    assert np.array_equal(a, b)
    # the first rows of a taller draw are the same bytes (counter-based)
    c = synth.weight(128, 96, seed=1, sigma=0.02, p=0.001, mult=20.0)
    assert np.array_equal(a, c[:64])
    x4 = synth.decode_x(4, K=128)
    x8 = synth.decode_x(8, K=128)
    assert np.array_equal(x4, x8[:4])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    f = rng.standard_normal(100000).astype(np.float32) * 10
    ours = synth.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_recipe_statistics():
    W = synth.weight(2000, 512, seed=1, sigma=0.02, p=0.001, mult=20.0)
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    big = np.abs(Wf) > 0.02 * 6
    assert 0.0004 < big.mean() < 0.0016
    assert abs(np.median(np.abs(Wf)) / 0.02 - 0.6745) < 0.02
    x = synth.bf16_bits_to_f32(synth.decode_x(16, K=4096)).astype(np.float64)
    rms = np.sqrt((x ** 2).mean(axis=1))
    assert np.all(np.abs(rms - 1) < 0.01)
    rows = synth.tiny_outlier_rows()
    assert len(set(rows.tolist())) == 4
    Wt = synth.bf16_bits_to_f32(synth.tiny_weight())
    rowmax = np.abs(Wt).max(axis=1)
    assert set(np.argsort(rowmax)[-4:].tolist()) == set(rows.tolist())
    s = synth.student_t3_row_scale(20000, seed=4)
    assert 0.5 < np.median(s) < 0.9 and s.max() > 10
