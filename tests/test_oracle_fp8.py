"""Pins of the oracle's fp8 copy (per-row E4M3 weights, per-token E4M3
activations, W8A8 product) against facts outside the oracle: a hand-derived
fixture, closed forms, brute-force nearest rounding on the E4M3 grid,
torch's own float8_e4m3fn cast, and numpy's float64 matmul."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_rows.txt")


def load_fixture():
    rows, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tag, *rest = line.split()
        if tag == "row":
            cur = {"name": rest[0]}
            rows.append(cur)
        elif tag == "x":
            cur["x"] = np.array([float(v) for v in rest], dtype=np.float32)
        elif tag == "scale":
            cur["scale"] = int(rest[0], 16)
        elif tag == "q":
            cur["q"] = np.array([int(v, 16) for v in rest], dtype=np.uint8)
    return rows


def test_hand_fixture():
    for r in load_fixture():
        xb = synth.f32_to_bf16_bits(r["x"])
        assert np.array_equal(synth.bf16_bits_to_f32(xb), r["x"]), r["name"]  # exact in bf16
        q, s = oracle.fp8_quantize(xb[None, :])
        assert int(s.view(np.uint32)[0]) == r["scale"], (r["name"], hex(int(s.view(np.uint32)[0])))
        assert np.array_equal(q[0], r["q"]), (r["name"], [hex(v) for v in q[0]])


E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
GRID = np.unique(np.abs(E4M3[np.isfinite(E4M3)]).astype(np.float64))  # 0 .. 448


def decode(q):
    return E4M3[q].astype(np.float64)


@pytest.fixture(scope="module")
def rows():
    W = synth.quant_weight(N=64, K=512, seed=3)
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    q, s = oracle.fp8_quantize(W)
    return W, Wf, q, s


def test_scale_closed_form_and_amax_code(rows):
    W, Wf, q, s = rows
    amax = np.abs(Wf).max(axis=1)
    # s is amax/448 rounded once to binary32: within half an ulp of the exact ratio
    exact = amax / 448.0
    ulp = np.spacing(s.astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(s.astype(np.float64) - exact) <= 0.5 * ulp)
    # the row maximum saturates to +-448: code 0x7e / 0xfe
    j = np.abs(Wf).argmax(axis=1)
    codes = q[np.arange(len(j)), j]
    assert np.all((codes & 0x7F) == 0x7E)
    assert np.all((codes >> 7) == (Wf[np.arange(len(j)), j] < 0))


def test_codes_are_the_nearest_grid_point(rows):
    """Brute force: each decoded |value| is the E4M3 grid point nearest to
    |x|/s (up to the rounding of 1/s and of x*(1/s), 2^-22 relative), ties
    to the even code; the sign follows x."""
    W, Wf, q, s = rows
    t = np.minimum(np.abs(Wf) / s[:, None].astype(np.float64), 448.0)
    d = np.abs(decode(q))
    dist = np.abs(GRID[None, None, :] - t[..., None])          # [N, K, 253]
    best = dist.min(axis=-1)
    got = np.abs(d - t)
    slack = t * 2.0 ** -22 + 1e-30
    assert np.all(got <= best + slack)
    # the sign bit is the sign of x, zeros included (-0 -> 0x80, as a cast keeps it)
    assert np.all((q >> 7) == np.signbit(Wf))


def test_round_trip_bound(rows):
    """|x - e4m3(q)*s| <= 2^-4 |x| (+ the subnormal step 2^-10 * s): half the
    relative spacing of a 3-bit mantissa."""
    W, Wf, q, s = rows
    back = decode(q) * s[:, None]
    err = np.abs(back - Wf)
    assert np.all(err <= 2.0 ** -4 * np.abs(Wf) + 2.0 ** -10 * s[:, None] * 1.0001)


def test_matches_torch_cast(rows):
    """The encode step equals torch's float8_e4m3fn cast of the scaled values."""
    W, Wf, q, s = rows
    r = (np.float32(1.0) / s).astype(np.float32)
    v = np.clip(synth.bf16_bits_to_f32(W) * r[:, None], -448, 448).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def test_zero_and_tiny_rows():
    W = np.zeros((2, 32), dtype=np.uint16)
    W[1, 5] = 0x0001  # the smallest bf16 subnormal
    q, s = oracle.fp8_quantize(W)
    assert s[0] == np.float32(1e-12) and not q[0].any()
    assert s[1] == np.float32(1e-12)   # amax/448 underflows the floor
    with pytest.raises(oracle.OracleError):
        bad = W.copy()
        bad[0, 0] = 0x7F80  # +Inf
        oracle.fp8_quantize(bad)


def test_product_matches_numpy():
    W, x = synth.tiny_weight(), synth.tiny_x()
    wq, ws = oracle.fp8_quantize(W)
    xq, xs = oracle.fp8_quantize(x)
    got = oracle.fp8_logits(xq, xs, wq, ws)
    ref = (decode(xq) * xs[:, None].astype(np.float64)) @ (decode(wq) * ws[:, None].astype(np.float64)).T
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    cols = np.array([0, 7, 511, 3])
    assert np.array_equal(oracle.fp8_logits(xq, xs, wq, ws, cols=cols), got[:, cols])
