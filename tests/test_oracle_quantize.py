"""Pins of the oracle's quantizer (CPU only).

Each test ties the oracle to something other than itself: a hand-derived
fixture, a closed form checked in exact rational arithmetic, an invariant of
the method, or an error bound that follows from the E2M1 grid spacing.  The
method is `_quantize_nvfp4` on the page
"vllm.model_executor.layers.quantization.online.lm_head"; its K % 16 rule is
the one `KNvfp4Static.create_weights` enforces on the page of
vllm/model_executor/layers/quantization/modelopt.py.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests import _fixtures


def test_hand_blocks_fixture():
    W, g, S, P = _fixtures.hand_blocks()
    packed, scales, glob = oracle.quantize(W)
    assert float(glob) == g
    assert np.array_equal(scales, S), (scales, S)
    assert np.array_equal(packed, P), (packed, P)


def _round_f32(x: Fraction) -> np.float32:
    """Correctly rounded binary32 of an exact rational (nearest, ties to even)."""
    c = np.float32(float(x))
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        err = abs(Fraction(float(cand)) - x)
        key = (err, int(np.array([cand]).view(np.uint32)[0]) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return best[1]


def test_global_scale_closed_form():
    rng = np.random.default_rng(3)
    amaxes = [0.0, 1e-30, 2688.0, 1.0, 3.171875, 448.0, 6.0]
    bits = rng.integers(0x0080, 0x7F7F, size=300, dtype=np.uint16)
    amaxes += [float(v) for v in synth.bf16_bits_to_f32(bits)]
    tiny = np.float32(1e-12)
    for a in amaxes:
        g, ig = oracle.global_scale(a)
        want = _round_f32(Fraction(float(np.float32(a))) / 2688)
        if want < tiny:
            want = tiny
        assert g == want, (a, g, want)
        assert ig == _round_f32(1 / Fraction(float(g)))
        if a > 2688 * 1e-12 * 2:
            # global * 2688 reproduces amax to within one binary32 rounding
            assert abs(float(g) * 2688 - a) <= a * 2.0 ** -23


def test_all_zero_weight():
    W = np.zeros((4, 32), dtype=np.uint16)
    packed, scales, g = oracle.quantize(W)
    assert g == np.float32(1e-12)
    assert not packed.any() and not scales.any()


def test_single_outlier():
    W = np.zeros((2, 32), dtype=np.uint16)
    W[1, 17] = synth.f32_to_bf16_bits(np.float32([-0.3]))[0]
    packed, scales, g = oracle.quantize(W)
    assert scales[1, 1] == 0x7E
    assert packed[1, 8] == (0xF << 4)  # element 17 is the high nibble of byte 8
    packed[1, 8] = 0
    scales[1, 1] = 0
    assert not packed.any() and not scales.any()


def _blocks_with_amax(W, packed, scales):
    Wf = synth.bf16_bits_to_f32(W)
    n, k = np.unravel_index(np.argmax(np.abs(Wf)), Wf.shape)
    code = (packed[n, k // 2] >> (4 * (k % 2))) & 15
    return Wf[n, k], scales[n, k // 16], code


@pytest.mark.parametrize("which", ["tiny", "random_t3", "negative_amax"])
def test_amax_block_invariant(which):
    """The block holding max|W| gets scale 448 (0x7e) and its element +-6."""
    if which == "tiny":
        W = synth.tiny_weight()
    elif which == "random_t3":
        W = synth.quant_weight(N=300, K=160, seed=11)
    else:
        W = synth.weight(64, 64, seed=5, sigma=1.0)
        Wf = synth.bf16_bits_to_f32(W).copy()
        Wf[10, 33] = -20.0
        W = synth.f32_to_bf16_bits(Wf)
    packed, scales, g = oracle.quantize(W)
    val, s, code = _blocks_with_amax(W, packed, scales)
    assert s == 0x7E
    assert code == (15 if val < 0 else 7)


def _halfstep(a):
    return np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))


@pytest.mark.parametrize("which", ["tiny", "decode_like", "t3"])
def test_round_trip_error_bound(which):
    """|x - dequant(x)| <= sf*g*(half the local grid step), sf a normal e4m3 scale.

    The grid steps are 0.5 below 2, 1 up to 4 and 2 up to 6; values beyond 6
    after scaling (the block scale rounds down by at most 1/16) are clamped
    to 6 and stay within 0.375 < 1 grid units.
    """
    if which == "tiny":
        W = synth.tiny_weight()
    elif which == "decode_like":
        W = synth.weight(256, 512, seed=9, sigma=0.02, p=0.01, mult=20.0)
    else:
        W = synth.quant_weight(N=256, K=512, seed=12)
    packed, scales, g = oracle.quantize(W)
    deq = oracle.dequant_rows(packed, scales, g)
    x = synth.bf16_bits_to_f32(W).astype(np.float64)
    sf = np.repeat(np.array([[oracle.e4m3_decode(int(b)) for b in row] for row in scales]),
                   16, axis=1)
    unit = sf * float(g)
    normal = sf >= 2.0 ** -6
    q = np.abs(x) / np.where(unit > 0, unit, 1)
    err = np.abs(x - deq)
    bound = unit * (_halfstep(q) + 1e-5)
    assert normal.mean() > 0.5
    assert np.all(err[normal] <= bound[normal])
    # and the dequantized tensor is a faithful copy in aggregate
    rel = np.linalg.norm(x - deq) / np.linalg.norm(x)
    assert rel < 0.15


def test_rows_are_independent_given_global():
    """Quantizing a row subset with the tensor's global scale equals the full run
    (the page's row chunking cannot change results)."""
    W = synth.quant_weight(N=97, K=96, seed=13)
    packed, scales, g = oracle.quantize(W)
    _, ig = oracle.global_scale(oracle.weight_amax(W))
    rows = np.array([96, 0, 50, 3, 3], dtype=np.int64)
    p2, s2 = oracle.quantize_rows(W, rows, g, ig)
    assert np.array_equal(p2, packed[rows])
    assert np.array_equal(s2, scales[rows])


def test_rejects_k_not_multiple_of_16_and_nonfinite():
    with pytest.raises(oracle.OracleError):
        oracle.quantize(np.zeros((2, 24), dtype=np.uint16))
    with pytest.raises(oracle.OracleError):
        oracle.quantize(np.zeros((0, 32), dtype=np.uint16))
    W = np.zeros((2, 32), dtype=np.uint16)
    W[1, 3] = 0x7F80  # +inf
    with pytest.raises(oracle.OracleError):
        oracle.quantize(W)
    W[1, 3] = 0x7FC1  # NaN
    with pytest.raises(oracle.OracleError):
        oracle.quantize(W)
