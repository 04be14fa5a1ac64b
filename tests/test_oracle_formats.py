"""Pins of the oracle's number formats (CPU only).

E2M1 codes and packing are pinned to the tables of the page
"vllm.model_executor.layers.quantization.online.lm_head" (`_quantize_nvfp4`),
kept as text fixtures in tests/golden/.  The E4M3 encoder and decoder are
pinned to torch's own float8_e4m3fn cast (an independent library routine),
exhaustively over every binary32 value in [0, 448].  The E2M1 rounding is
pinned to a brute-force nearest-grid-point search.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import _fixtures

E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def test_code_map_matches_page_table():
    table = _fixtures.code_map()
    assert [c for _, c, _ in table] == list(range(8))
    for doubled, code, mag in table:
        assert doubled == int(mag * 2)
        assert oracle.e2m1_code(mag) == code
        assert oracle.e2m1_decode(code) == mag
        if mag > 0:
            assert oracle.e2m1_code(-mag) == code | 8
            assert oracle.e2m1_decode(code | 8) == -mag
    # a value that is zero carries no sign bit, even as -0.0
    assert oracle.e2m1_code(-0.0) == 0
    # off-grid values are rejected by the code lookup
    assert oracle.e2m1_code(2.5) == 0xFF


def test_packing_low_nibble_first():
    """Decode direction: byte -> (element 2j, element 2j+1) with scale 1, global 1."""
    for v0, v1, byte in _fixtures.packing():
        packed = np.array([[byte]], dtype=np.uint8)
        scales = np.array([[0x38]], dtype=np.uint8)  # e4m3 1.0
        w = oracle.dequant_rows(packed, scales, np.float32(1.0))
        assert w.tolist() == [[v0, v1]], (hex(byte), w)


def test_e4m3_decode_all_bytes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    ours = np.array([oracle.e4m3_decode(int(c)) for c in codes], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


@pytest.mark.parametrize("chunk", range(0, 17))
def test_e4m3_encode_exhaustive_vs_torch(chunk):
    """Every binary32 bit pattern in [0, 448], 17 chunks of 2^26 patterns."""
    top = int(np.array([448.0], dtype=np.float32).view(np.uint32)[0])
    lo = chunk << 26
    hi = min((chunk + 1) << 26, top + 1)
    if lo >= hi:
        pytest.skip("past 448")
    bits = np.arange(lo, hi, dtype=np.uint32)
    t = bits.view(np.float32)
    ours = oracle.e4m3_encode_array(t)
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(t[i]), int(ours[i]), int(ref[i])) for i in bad[:5]]


def test_e4m3_encode_ties_to_even_mantissa():
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)], dtype=np.float64)
    for c in range(0x7E):
        mid = np.float32((vals[c] + vals[c + 1]) / 2)  # exact: few significant bits
        assert float(mid) == (vals[c] + vals[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == even
        assert oracle.e4m3_encode(float(np.nextafter(mid, np.float32(1e9)))) == c + 1
        assert oracle.e4m3_encode(float(np.nextafter(mid, np.float32(0)))) == c


def _brute_force_round(q: np.ndarray) -> np.ndarray:
    a = np.abs(q.astype(np.float64))
    d = np.abs(a[:, None] - E2M1_MAGS[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equally near grid points take the even code (index)
    idx = np.where(cand[:, ::2].any(axis=1),
                   np.argmax(cand & (np.arange(8) % 2 == 0), axis=1),
                   np.argmax(cand, axis=1))
    return np.copysign(E2M1_MAGS[idx], q).astype(np.float32)


def test_e2m1_round_bruteforce():
    rng = np.random.default_rng(7)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    pts = [mids, np.nextafter(mids, np.float32(10)), np.nextafter(mids, np.float32(0)),
           E2M1_MAGS.astype(np.float32), np.linspace(0, 6, 200001, dtype=np.float32),
           rng.uniform(0, 6, 500000).astype(np.float32), np.float32([6.0, 0.0])]
    q = np.concatenate(pts)
    q = np.concatenate([q, -q])
    ours = oracle.e2m1_round_array(q)
    ref = _brute_force_round(q)
    assert np.array_equal(ours, ref)
    assert np.array_equal(np.signbit(ours), np.signbit(q))


def test_e2m1_negative_value_rounding_to_zero_has_code_zero():
    v = oracle.e2m1_round(-0.1)
    assert v == 0.0 and np.signbit(v)
    assert oracle.e2m1_code(v) == 0
