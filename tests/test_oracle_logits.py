"""Pins of the oracle's W4A16 product (CPU only).

The product is the weight-only NVFP4 linear of `CompressedTensorsW4A16Fp4`
(page "vllm.model_executor.layers.quantization.compressed_tensors.schemes"):
logits = x . W^T with W = e2m1(code) * f32(block scale) * global, the global
scale being the amax/2688 dequant multiplier (page of
vllm/model_executor/layers/quantization/modelopt.py, `KNvfp4Static.process`).
"""
import numpy as np
import torch

import oracle
import synth
from tests import _fixtures


def test_logits_equal_numpy_matmul_of_dequant():
    W = synth.tiny_weight()
    x = synth.tiny_x()
    packed, scales, g = oracle.quantize(W)
    got = oracle.logits(x, packed, scales, g)
    xd = synth.bf16_bits_to_f32(x).astype(np.float64)
    ref = xd @ oracle.dequant_rows(packed, scales, g).T
    assert got.shape == (4, 512)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_logits_column_subset():
    W = synth.quant_weight(N=200, K=64, seed=21)
    x = synth.decode_x(3, K=64)
    packed, scales, g = oracle.quantize(W)
    full = oracle.logits(x, packed, scales, g)
    cols = np.array([199, 0, 7, 7, 100], dtype=np.int64)
    sub = oracle.logits(x, packed, scales, g, cols=cols)
    assert np.array_equal(sub, full[:, cols])


def test_logits_brute_force_from_page_tables():
    """Pure-Python decode from the page's code table and torch's e4m3 cast."""
    rng = np.random.default_rng(5)
    N, K, M = 3, 32, 2
    packed = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = np.array(rng.choice([0x00, 0x01, 0x30, 0x38, 0x39, 0x55, 0x7E], size=(N, K // 16)),
                      dtype=np.uint8)
    g = np.float32(0.0123)
    x = synth.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    mag = {code: m for _, code, m in _fixtures.code_map()}
    sf = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).double().numpy()
    xd = synth.bf16_bits_to_f32(x).astype(np.float64)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                byte = int(packed[n, k // 2])
                code = byte & 15 if k % 2 == 0 else byte >> 4
                w = mag[code & 7] * (-1.0 if code & 8 else 1.0) * sf[n, k // 16] * float(g)
                acc += xd[m, k] * w
            want[m, n] = acc
    got = oracle.logits(x, packed, scales, g)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
