"""Pins of the oracle's W4A4 parts: the 128x4-interleaved block-scale layout
against hand-derived byte positions, and the W4A4 product against numpy's
float64 matmul of the separately pinned quantize/dequant steps and against
the W4A16 product where x is exactly representable."""
import numpy as np

import oracle
import synth


def test_swizzle_layout_hand_positions():
    """130 rows (two 128-row bands, the second ragged) x 8 columns (two
    4-column groups): byte (r, c) of the source lands where the layout of
    `swizzle_blockscale` puts it; worked out by hand from its
    [N/128][4][32][C/4][4] -> [N/128][C/4][32][4][4] reordering."""
    N, C = 130, 8
    src = np.zeros((N, C), dtype=np.uint8)
    cases = {  # (row, col): expected flat position
        (0, 0): 0, (0, 1): 1, (0, 3): 3, (1, 0): 16, (31, 0): 496, (32, 0): 4,
        (33, 2): 22, (96, 3): 15, (0, 4): 512, (127, 7): 1023, (128, 0): 1024,
        (129, 5): 1553,
    }
    for i, (rc, _) in enumerate(cases.items()):
        src[rc] = i + 1
    out = oracle.swizzle_scales(src)
    assert out.size == 256 * 8
    for i, (rc, pos) in enumerate(cases.items()):
        assert out[pos] == i + 1, (rc, pos, int(np.argwhere(out == i + 1)[0, 0]))
    assert np.count_nonzero(out) == len(cases)     # padding rows and other bytes are zero
    # every source byte appears exactly once
    full = (np.arange(N * C) % 251 + 1).astype(np.uint8).reshape(N, C)
    got = oracle.swizzle_scales(full)
    assert sorted(got[got != 0].tolist()) == sorted(full.reshape(-1).tolist())


def test_product_matches_numpy():
    W, x = synth.tiny_weight(), synth.tiny_x()
    p, s, gw = oracle.quantize(W)
    amax = float(np.abs(synth.bf16_bits_to_f32(x)).max())
    gx, igx = oracle.global_scale(amax)
    xp, xs = oracle.quantize_rows(x, np.arange(x.shape[0]), gx, igx)
    ref = oracle.dequant_rows(xp, xs, gx) @ oracle.dequant_rows(p, s, gw).T
    got = oracle.w4a4_logits(x, gx, p, s, gw)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)
    cols = np.array([5, 0, 511])
    assert np.array_equal(oracle.w4a4_logits(x, gx, p, s, gw, cols=cols), got[:, cols])


def test_exact_activations_match_w4a16():
    """x made of E2M1 grid values with every block maximum 6 and an input
    global of 1 is quantized losslessly (scale exactly 1), so the W4A4
    logits equal the W4A16 logits."""
    rng = np.random.default_rng(1)
    K, M = 256, 3
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    xf = grid[rng.integers(0, 8, (M, K))] * rng.choice([-1.0, 1.0], (M, K))
    xf[:, ::16] = 6.0
    x = synth.f32_to_bf16_bits(xf.astype(np.float32))
    W = synth.quant_weight(N=300, K=K, seed=2)
    p, s, gw = oracle.quantize(W)
    assert np.array_equal(oracle.w4a4_logits(x, 1.0, p, s, gw), oracle.logits(x, p, s, gw))
